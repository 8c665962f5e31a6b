// TTT-MLP forward on the tensor cores (bf16 inputs, d = 64, hidden m = 256,
// chunk b a multiple of 16): one CTA of 16 warps per (batch row, head).
//
// Method ("Test-Time Training (TTT) guide", section 3: two layers, hidden 4x
// the input, GELU; "5 · TestingTime 训练与长上下文", section 1.1: gradients at
// the chunk-start weights, dual form). Per 16-token tile of a chunk, with
// W1a, W2a the chunk-start weights and W1, W2 the running ones:
//   U = K W1a,  A = gelu(U),  P = gelu'(U)
//   G = A W2a - V,  D = (G W2a^T) .* P
//   Hq = Q W1 - eta tril(Q K^T) D,  Aq = gelu(Hq)
//   Z = Aq W2 - eta tril(Aq A^T) G
//   W1 -= eta K^T D,  W2 -= eta A^T G
// (for b = 16 every tile is a chunk and W1a = W1, W2a = W2). gelu is the tanh
// form of Hendrycks and Gimpel (2016), evaluated with the tanh.approx.f32
// instruction.
//
// Layout. The fp32 weights live in registers as mma.sync accumulator
// fragments, split by hidden unit: warp w owns W1[:, 16w:16w+16] and
// W2[16w:16w+16, :] (64 floats per lane), and updates them with the chunk's
// rank-16 gradient products. bf16 copies of W1 and W2 sit in shared memory
// (rewritten after every update, 128-byte XOR swizzle), so every product reads
// whatever fragment layout it needs with ldmatrix, transposed or not. Q, K, V
// tiles arrive by TMA, double-buffered. Products over the hidden dimension
// (G, Z) are split across warps by hidden quarter and summed through shared
// memory; tril(Aq A^T) is linear in its hidden terms, so each quarter applies
// its own part of it to G before that sum.
#include "kernels.h"
#include "mlp_frag.cuh"
#include "ttt_device.cuh"

namespace ttt {
namespace {

using namespace mlpf;

constexpr int kD = 64;
constexpr int kM = 256;
constexpr int kTile = 16;
constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kTileBytes = kTile * kD * 2;          // 2 KB
constexpr int kRowM = kM * 2;                        // 512-byte rows of [.][256] bf16
// shared memory map (bytes from a 1024-aligned base)
constexpr int kQKV = 0;                              // [2 stages][Q, K, V] tiles
constexpr int kW1b = kQKV + 2 * 3 * kTileBytes;      // W1 running, bf16 [64][256]
constexpr int kW2b = kW1b + kD * kRowM;              // W2 running, bf16 [256][64]
constexpr int kAb = kW2b + kM * 128;                 // A, bf16 [16][256]
constexpr int kAqb = kAb + kTile * kRowM;            // Aq
constexpr int kGb = kAqb + kTile * kRowM;            // G, bf16 [16][64]
constexpr int kSb = kGb + kTile * 128;               // tril(Q K^T), bf16 [16][16] in 128-byte rows
constexpr int kPart = kSb + kTile * 128;             // partial sums, fp32: G or Z [4][16][kPad]
constexpr int kPad = 68;                             // fp32 row stride of the partial buffers
constexpr int kBar = kPart + 4 * kTile * kPad * 4;   // 2 mbarriers
constexpr int kBaseBytes = kBar + 64;
constexpr int kW1s = kBaseBytes;                     // chunk-start copies (b > 16 only)
constexpr int kW2s = kW1s + kD * kRowM;
constexpr int kSnapBytes = kD * kRowM + kM * 128;

enum : int { kWhereMlpLoad = 12 };

__global__ void __launch_bounds__(kThreads, 1)
    mlp_mma_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                   const __grid_constant__ CUtensorMap mv, MlpParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + kBar);
  const uint32_t s0 = smem_u32(sm);
  const bool snap = p.b > kTile;  // separate chunk-start copies
  uint8_t* W1s = snap ? sm + kW1s : sm + kW1b;
  uint8_t* W2s = snap ? sm + kW2s : sm + kW2b;
  float* part = reinterpret_cast<float*>(sm + kPart);

  const int unit = blockIdx.x;
  const int h = unit % p.H;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, tg = lane & 3;
  const float eta = p.eta[h];
  const int n_tiles = (p.T + kTile - 1) / kTile;

  if (tid == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    fence_barrier_init();
  }
  // fp32 masters (C fragments): W1[:, 16w:16w+16] as 4 m-tiles (i) x 2 n-tiles (hidden),
  // W2[16w:16w+16, :] as 8 n-tiles (j).
  float w1[4][2][4], w2[8][4];
  {
    const float* W10 = p.W1_0 + static_cast<size_t>(h) * kD * kM;
    const float* W20 = p.W2_0 + static_cast<size_t>(h) * kM * kD;
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int i = 16 * mt + g, c = 16 * warp + 8 * nt + 2 * tg;
        w1[mt][nt][0] = W10[i * kM + c];
        w1[mt][nt][1] = W10[i * kM + c + 1];
        w1[mt][nt][2] = W10[(i + 8) * kM + c];
        w1[mt][nt][3] = W10[(i + 8) * kM + c + 1];
      }
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int r = 16 * warp + g, c = 8 * nt + 2 * tg;
      w2[nt][0] = W20[r * kD + c];
      w2[nt][1] = W20[r * kD + c + 1];
      w2[nt][2] = W20[(r + 8) * kD + c];
      w2[nt][3] = W20[(r + 8) * kD + c + 1];
    }
  }
// bf16 copies of this warp's slices of the running weights.
#define TTT_STORE_W1(dst)                                                          \
  do {                                                                              \
    _Pragma("unroll") for (int mt = 0; mt < 4; ++mt)                               \
      _Pragma("unroll") for (int nt = 0; nt < 2; ++nt) {                           \
        const int ch = 2 * warp + nt;                                               \
        *reinterpret_cast<uint32_t*>((dst) + swz(16 * mt + g, ch, kRowM) + 4 * tg) =  \
            pack_bf16(w1[mt][nt][0], w1[mt][nt][1]);                                 \
        *reinterpret_cast<uint32_t*>((dst) + swz(16 * mt + g + 8, ch, kRowM) + 4 * tg) = \
            pack_bf16(w1[mt][nt][2], w1[mt][nt][3]);                                 \
      }                                                                             \
  } while (0)
#define TTT_STORE_W2(dst)                                                          \
  do {                                                                              \
    _Pragma("unroll") for (int nt = 0; nt < 8; ++nt) {                             \
      *reinterpret_cast<uint32_t*>((dst) + swz(16 * warp + g, nt, 128) + 4 * tg) =  \
          pack_bf16(w2[nt][0], w2[nt][1]);                                          \
      *reinterpret_cast<uint32_t*>((dst) + swz(16 * warp + g + 8, nt, 128) + 4 * tg) = \
          pack_bf16(w2[nt][2], w2[nt][3]);                                          \
    }                                                                               \
  } while (0)
  TTT_STORE_W1(sm + kW1b);
  TTT_STORE_W2(sm + kW2b);
  if (snap) {
    TTT_STORE_W1(W1s);
    TTT_STORE_W2(W2s);
  }
  __syncthreads();

  auto load_tile = [&mq, &mk, &mv, &full, sm, unit](int u) {
    const int s = u & 1;
    uint8_t* st = sm + kQKV + s * 3 * kTileBytes;
    mbar_arrive_expect_tx(&full[s], 3 * kTileBytes);
    tma_load_3d(st, &mq, &full[s], 0, u * kTile, unit);
    tma_load_3d(st + kTileBytes, &mk, &full[s], 0, u * kTile, unit);
    tma_load_3d(st + 2 * kTileBytes, &mv, &full[s], 0, u * kTile, unit);
  };
  if (tid == 0 && n_tiles > 0 && p.inject_stall != 1) {  // test hook: the loads never start
    prefetch_tmap(&mq);
    prefetch_tmap(&mk);
    prefetch_tmap(&mv);
    load_tile(0);
  }

  const uint32_t W1b = s0 + kW1b, W2b = s0 + kW2b, W1sa = smem_u32(W1s), W2sa = smem_u32(W2s);
  const uint32_t Ab = s0 + kAb, Aqb = s0 + kAqb, Gb = s0 + kGb, Sb = s0 + kSb;
  bool ok = true;

  for (int u = 0; u < n_tiles; ++u) {
    const int s = u & 1;
    const uint32_t sQ = s0 + kQKV + s * 3 * kTileBytes, sK = sQ + kTileBytes;
    const uint8_t* sVp = sm + kQKV + s * 3 * kTileBytes + 2 * kTileBytes;
    // Every thread waits for this tile's data (bounded); the next tile's loads go
    // into the other stage, whose last readers finished before the previous
    // tile's final barrier.
    if (!mbar_wait_bounded(&full[s], (u >> 1) & 1, p.timeout_ns)) {
      if (lane == 0) report_error(p.status, TTT_ERR_TIMEOUT, kWhereMlpLoad, unit);
      ok = false;
    }
    // Every thread's reads of the other stage (the previous tile) are complete at the
    // barrier below; the proxy fence also orders them before the async-proxy TMA write
    // that refills that stage next.
    fence_proxy_async_smem();
    if (__syncthreads_or(!ok)) {
      // This tile's load may still be in flight: let it land before the CTA exits.
      if (tid == 0) (void)mbar_wait_bounded(&full[s], (u >> 1) & 1, p.timeout_ns);
      break;
    }
    if (tid == 0 && u + 1 < n_tiles) load_tile(u + 1);
    const bool chunk_end = ((u + 1) * kTile) % p.b == 0 || u + 1 == n_tiles;

    // (1) U = K W1a for hidden [16w, 16w+16); A, P.  Warp 0 also forms tril(Q K^T).
    float cu[2][4] = {}, cp[2][4];
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      uint32_t a[4], b[4];
      ldA(a, sK, 128, 0, 2 * ks, lane);
      ldBT(b, W1sa, kRowM, 16 * ks, 2 * warp, lane);
      mma2(cu, a, b);
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) gelu2(cu[nt][r], cu[nt][r], cp[nt][r]);
    st_tile(sm + kAb, kRowM, 0, warp, cu, lane);
    if (warp < 2) {  // warp nt forms columns [8nt, 8nt + 8) of S
      const int nt = warp;
      float cs[4] = {};
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        uint32_t a[4], b[4];
        ldA(a, sQ, 128, 0, 2 * ks, lane);
        ldB(b, sK, 128, 0, 2 * ks, lane);
        const uint32_t bn[2] = {nt ? b[2] : b[0], nt ? b[3] : b[1]};  // selects: no local copy of b
        mma_bf16_16816(cs, a, bn);
      }
      const int c = 8 * nt + 2 * tg;  // keep column <= row (update, then read)
      if (c > g) cs[0] = 0.f;
      if (c + 1 > g) cs[1] = 0.f;
      if (c > g + 8) cs[2] = 0.f;
      if (c + 1 > g + 8) cs[3] = 0.f;
      *reinterpret_cast<uint32_t*>(sm + kSb + swz(g, nt, 128) + 4 * tg) = pack_bf16(cs[0], cs[1]);
      *reinterpret_cast<uint32_t*>(sm + kSb + swz(g + 8, nt, 128) + 4 * tg) = pack_bf16(cs[2], cs[3]);
    }
    __syncthreads();

    // (2) G partials: warp -> value columns [16(w&3), +16), hidden quarter w>>2.
    {
      const int np = warp & 3, kq = warp >> 2;
      float cg[2][4] = {};
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        uint32_t a[4], b[4];
        ldA(a, Ab, kRowM, 0, 8 * kq + 2 * ks, lane);
        ldBT(b, W2sa, 128, 64 * kq + 16 * ks, 2 * np, lane);
        mma2(cg, a, b);
      }
      float* dst = part + kq * kTile * kPad;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int c = 16 * np + 8 * nt + 2 * tg;
        *reinterpret_cast<float2*>(dst + g * kPad + c) = make_float2(cg[nt][0], cg[nt][1]);
        *reinterpret_cast<float2*>(dst + (g + 8) * kPad + c) = make_float2(cg[nt][2], cg[nt][3]);
      }
    }
    __syncthreads();
    // G = sum of the quarters - V, fp32 and bf16.
    {
      const int t = tid >> 5, j = (tid & 31) * 2;
      float2 acc = make_float2(0.f, 0.f);
#pragma unroll
      for (int kq = 0; kq < 4; ++kq) {
        const float2 v = *reinterpret_cast<const float2*>(part + kq * kTile * kPad + t * kPad + j);
        acc.x += v.x;
        acc.y += v.y;
      }
      const uint32_t vv = *reinterpret_cast<const uint32_t*>(sVp + swz(t, j >> 3, 128) + (j & 7) * 2);
      acc.x -= bf16_lo(vv);
      acc.y -= bf16_hi(vv);
      *reinterpret_cast<uint32_t*>(sm + kGb + swz(t, j >> 3, 128) + (j & 7) * 2) = pack_bf16(acc.x, acc.y);
    }
    __syncthreads();

    // (3) D = (G W2a^T) .* P for hidden [16w, +16);  W2 -= eta A^T G (this warp's rows).
    uint32_t bd[4];
    {
      float cd[2][4] = {};
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        uint32_t a[4], b[4];
        ldA(a, Gb, 128, 0, 2 * ks, lane);
        ldB(b, W2sa, 128, 16 * warp, 2 * ks, lane);
        mma2(cd, a, b);
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) cd[nt][r] *= cp[nt][r];
      // D as the B operand (k = t, n = hidden) of S D and K^T D: the transposed 8 x 8
      // blocks of its C fragment, in registers (no other warp reads this warp's D).
      bd[0] = movm_t(pack_bf16(cd[0][0], cd[0][1]));
      bd[1] = movm_t(pack_bf16(cd[0][2], cd[0][3]));
      bd[2] = movm_t(pack_bf16(cd[1][0], cd[1][1]));
      bd[3] = movm_t(pack_bf16(cd[1][2], cd[1][3]));

      uint32_t a[4];
      ldAT(a, Ab, kRowM, 0, 2 * warp, lane);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t b[4];
        ldBT(b, Gb, 128, 0, 2 * q, lane);
        float acc[2][4] = {};
        mma2(acc, a, b);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int r = 0; r < 4; ++r) w2[2 * q + nt][r] = fmaf(-eta, acc[nt][r], w2[2 * q + nt][r]);
      }
    }

    // (4) Hq = Q W1 - eta tril(Q K^T) D, Aq = gelu(Hq);  W1 -= eta K^T D (this warp's columns).
    {
      float ch[2][4] = {}, cs[2][4] = {};
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        uint32_t a[4], b[4];
        ldA(a, sQ, 128, 0, 2 * ks, lane);
        ldBT(b, W1b, kRowM, 16 * ks, 2 * warp, lane);
        mma2(ch, a, b);
      }
      {
        uint32_t a[4];
        ldA(a, Sb, 128, 0, 0, lane);
        mma2(cs, a, bd);
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) ch[nt][r] = gelu1(fmaf(-eta, cs[nt][r], ch[nt][r]));
      st_tile(sm + kAqb, kRowM, 0, warp, ch, lane);

#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        uint32_t a[4];
        ldAT(a, sK, 128, 0, 2 * mt, lane);
        float acc[2][4] = {};
        mma2(acc, a, bd);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int r = 0; r < 4; ++r) w1[mt][nt][r] = fmaf(-eta, acc[nt][r], w1[mt][nt][r]);
      }
    }
    // Columns [16w, +16) of the W1 copies are read by this warp alone (U, Hq): rewrite them now.
    __syncwarp();
    TTT_STORE_W1(sm + kW1b);
    if (snap && chunk_end) TTT_STORE_W1(W1s);
    __syncthreads();  // Aq complete
    // (5) Z partials: warp -> value columns [16(w&3), +16), hidden quarter kq = w>>2:
    //     Aq_kq W2_kq - eta tril(Aq_kq A_kq^T) G, the second term by the quarter's own
    //     16 x 16 block of tril(Aq A^T) (the four quarters' blocks sum to the whole).
    {
      const int np = warp & 3, kq = warp >> 2;
      float cz[2][4] = {}, csa[2][4] = {};
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        uint32_t a[4], b[4], ba[4];
        ldA(a, Aqb, kRowM, 0, 8 * kq + 2 * ks, lane);
        ldBT(b, W2b, 128, 64 * kq + 16 * ks, 2 * np, lane);
        ldB(ba, Ab, kRowM, 0, 8 * kq + 2 * ks, lane);
        mma2(cz, a, b);
        mma2(csa, a, ba);
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {  // keep t2 <= t, scale by -eta
        const int c = 8 * nt + 2 * tg;
        csa[nt][0] = c > g ? 0.f : -eta * csa[nt][0];
        csa[nt][1] = c + 1 > g ? 0.f : -eta * csa[nt][1];
        csa[nt][2] = c > g + 8 ? 0.f : -eta * csa[nt][2];
        csa[nt][3] = c + 1 > g + 8 ? 0.f : -eta * csa[nt][3];
      }
      // The C fragment of the 16 x 16 block is the A fragment (m = t, k = t2) of the next product.
      const uint32_t sa[4] = {pack_bf16(csa[0][0], csa[0][1]), pack_bf16(csa[0][2], csa[0][3]),
                              pack_bf16(csa[1][0], csa[1][1]), pack_bf16(csa[1][2], csa[1][3])};
      uint32_t bg[4];
      ldBT(bg, Gb, 128, 0, 2 * np, lane);
      mma2(cz, sa, bg);
      float* dst = part + kq * kTile * kPad;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int c = 16 * np + 8 * nt + 2 * tg;
        *reinterpret_cast<float2*>(dst + g * kPad + c) = make_float2(cz[nt][0], cz[nt][1]);
        *reinterpret_cast<float2*>(dst + (g + 8) * kPad + c) = make_float2(cz[nt][2], cz[nt][3]);
      }
    }
    __syncthreads();  // every read of the running W2 copy is done; the Z partials are written

    TTT_STORE_W2(sm + kW2b);
    if (snap && chunk_end) TTT_STORE_W2(W2s);
    // Z = sum of the quarters, written for the rows inside the sequence.
    {
      const int t = tid >> 5, j = (tid & 31) * 2;
      float2 z = make_float2(0.f, 0.f);
#pragma unroll
      for (int kq = 0; kq < 4; ++kq) {
        const float2 v = *reinterpret_cast<const float2*>(part + kq * kTile * kPad + t * kPad + j);
        z.x += v.x;
        z.y += v.y;
      }
      const int tt = u * kTile + t;
      if (tt < p.T) {
        __nv_bfloat16* Z = static_cast<__nv_bfloat16*>(p.Z) + (static_cast<size_t>(unit) * p.T + tt) * kD + j;
        *reinterpret_cast<uint32_t*>(Z) = pack_bf16(z.x, z.y);
      }
    }
    // No barrier here: the next tile first meets at its start barrier, and the buffer read
    // above (part) is written again only after that.
  }
  // Final state.
  float* W1o = p.W1_out + static_cast<size_t>(unit) * kD * kM;
  float* W2o = p.W2_out + static_cast<size_t>(unit) * kM * kD;
#pragma unroll
  for (int mt = 0; mt < 4; ++mt)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int i = 16 * mt + g, c = 16 * warp + 8 * nt + 2 * tg;
      *reinterpret_cast<float2*>(W1o + i * kM + c) = make_float2(w1[mt][nt][0], w1[mt][nt][1]);
      *reinterpret_cast<float2*>(W1o + (i + 8) * kM + c) = make_float2(w1[mt][nt][2], w1[mt][nt][3]);
    }
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    const int r = 16 * warp + g, c = 8 * nt + 2 * tg;
    *reinterpret_cast<float2*>(W2o + r * kD + c) = make_float2(w2[nt][0], w2[nt][1]);
    *reinterpret_cast<float2*>(W2o + (r + 8) * kD + c) = make_float2(w2[nt][2], w2[nt][3]);
  }
}

// Shared memory of mlp_mma16_kernel (b = 16: every tile is a chunk).
namespace pipe {
constexpr int kQKV = 0;                                // [2 stages][Q, K, V] tiles
constexpr int kW1b = kQKV + 2 * 3 * kTileBytes;        // W1 running, bf16 [64][256]
constexpr int kW2Bytes = kM * 128;
constexpr int kW2b = kW1b + kD * kRowM;                // W2 running, bf16 [2][256][64]: tile u reads copy u & 1
constexpr int kABytes = kTile * kRowM;
constexpr int kAb = kW2b + 2 * kW2Bytes;               // A, bf16 [2][16][256]: tile u's in copy u & 1
constexpr int kAqb = kAb + 2 * kABytes;                // Aq, bf16 [16][256]
constexpr int kGb = kAqb + kABytes;                    // G, bf16 [16][64]
constexpr int kSb = kGb + kTile * 128;                 // tril(Q K^T), bf16 [16][16] in 128-byte rows
constexpr int kPartG = kSb + kTile * 128;              // G partials, fp32 [4][16][kPad]
constexpr int kPartZ = kPartG + 4 * kTile * kPad * 4;  // Z partials, fp32 [4][16][kPad]
constexpr int kBar = kPartZ + 4 * kTile * kPad * 4;    // 2 mbarriers
constexpr int kBytes = kBar + 64;
static_assert(kBytes + 1024 <= 227 * 1024, "one CTA per SM");
}  // namespace pipe

// TTT-MLP forward for b = 16, software-pipelined over tiles. The Z of tile u depends
// on nothing the next tile needs, and tile u + 1's U, A, P and tril(Q K^T) depend on
// tile u only through the W1 update. So each tile runs in four barrier-separated
// phases:
//   (G)  G partials of tile u          +  the Z sum of tile u - 1
//   (R)  G = sum of the partials - V
//   (DH) D, the W2 update, Hq, Aq, the W1 update (as in mlp_mma_kernel)
//   (N)  U, A, P, tril(QK^T) of tile u + 1  +  the Z partials of tile u  +  tile u's
//        new W2 into the other bf16 copy
// (six in mlp_mma_kernel). A and W2 have two bf16 copies, by tile parity, and the G
// and Z partials separate buffers, so that work of neighbouring tiles in one phase
// touches disjoint data.
__global__ void __launch_bounds__(kThreads, 1)
    mlp_mma16_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                     const __grid_constant__ CUtensorMap mv, MlpParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + pipe::kBar);
  const uint32_t s0 = smem_u32(sm);
  float* partG = reinterpret_cast<float*>(sm + pipe::kPartG);
  float* partZ = reinterpret_cast<float*>(sm + pipe::kPartZ);

  const int unit = blockIdx.x;
  const int h = unit % p.H;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, tg = lane & 3;
  const float eta = p.eta[h];
  const int n_tiles = (p.T + kTile - 1) / kTile;

  if (tid == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    fence_barrier_init();
  }
  float w1[4][2][4], w2[8][4];
  {
    const float* W10 = p.W1_0 + static_cast<size_t>(h) * kD * kM;
    const float* W20 = p.W2_0 + static_cast<size_t>(h) * kM * kD;
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int i = 16 * mt + g, c = 16 * warp + 8 * nt + 2 * tg;
        w1[mt][nt][0] = W10[i * kM + c];
        w1[mt][nt][1] = W10[i * kM + c + 1];
        w1[mt][nt][2] = W10[(i + 8) * kM + c];
        w1[mt][nt][3] = W10[(i + 8) * kM + c + 1];
      }
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int r = 16 * warp + g, c = 8 * nt + 2 * tg;
      w2[nt][0] = W20[r * kD + c];
      w2[nt][1] = W20[r * kD + c + 1];
      w2[nt][2] = W20[(r + 8) * kD + c];
      w2[nt][3] = W20[(r + 8) * kD + c + 1];
    }
  }
  TTT_STORE_W1(sm + pipe::kW1b);
  TTT_STORE_W2(sm + pipe::kW2b);
  __syncthreads();

  int issued = 0;  // tiles whose loads thread 0 has issued
  auto load_tile = [&](int u) {
    const int s = u & 1;
    uint8_t* st = sm + pipe::kQKV + s * 3 * kTileBytes;
    mbar_arrive_expect_tx(&full[s], 3 * kTileBytes);
    tma_load_3d(st, &mq, &full[s], 0, u * kTile, unit);
    tma_load_3d(st + kTileBytes, &mk, &full[s], 0, u * kTile, unit);
    tma_load_3d(st + 2 * kTileBytes, &mv, &full[s], 0, u * kTile, unit);
    issued = u + 1;
  };
  if (tid == 0 && n_tiles > 0 && p.inject_stall != 1) {  // test hook: the loads never start
    prefetch_tmap(&mq);
    prefetch_tmap(&mk);
    prefetch_tmap(&mv);
    load_tile(0);
    if (n_tiles > 1) load_tile(1);
  }

  const uint32_t W1b = s0 + pipe::kW1b, Aqb = s0 + pipe::kAqb, Gb = s0 + pipe::kGb, Sb = s0 + pipe::kSb;
  float cp[2][4];  // gelu'(U) of the tile whose U ran last

  // Every thread waits for tile v's data (bounded).
  auto wait_tile = [&](int v) -> bool {
    const bool mine = mbar_wait_bounded(&full[v & 1], (v >> 1) & 1, p.timeout_ns);
    if (!mine) report_error(p.status, TTT_ERR_TIMEOUT, kWhereMlpLoad, unit);
    return mine;
  };
  // U = K W1 for this warp's hidden units [16w, +16), A = gelu(U) into copy v & 1, cp = gelu'(U);
  // warps 0 and 1 form one n-tile each of tril(Q K^T).
  auto phase_u = [&](int v) {
    const int s = v & 1;
    const uint32_t sQ = s0 + pipe::kQKV + s * 3 * kTileBytes, sK = sQ + kTileBytes;
    float cu[2][4] = {};
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      uint32_t a[4], b[4];
      ldA(a, sK, 128, 0, 2 * ks, lane);
      ldBT(b, W1b, kRowM, 16 * ks, 2 * warp, lane);
      mma2(cu, a, b);
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) gelu2(cu[nt][r], cu[nt][r], cp[nt][r]);
    st_tile(sm + pipe::kAb + s * pipe::kABytes, kRowM, 0, warp, cu, lane);
    if (warp < 2) {
      const int nt = warp;
      float cs[4] = {};
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        uint32_t a[4], b[4];
        ldA(a, sQ, 128, 0, 2 * ks, lane);
        ldB(b, sK, 128, 0, 2 * ks, lane);
        const uint32_t bn[2] = {nt ? b[2] : b[0], nt ? b[3] : b[1]};  // selects: no local copy of b
        mma_bf16_16816(cs, a, bn);
      }
      const int c = 8 * nt + 2 * tg;  // keep column <= row (update, then read)
      if (c > g) cs[0] = 0.f;
      if (c + 1 > g) cs[1] = 0.f;
      if (c > g + 8) cs[2] = 0.f;
      if (c + 1 > g + 8) cs[3] = 0.f;
      *reinterpret_cast<uint32_t*>(sm + pipe::kSb + swz(g, nt, 128) + 4 * tg) = pack_bf16(cs[0], cs[1]);
      *reinterpret_cast<uint32_t*>(sm + pipe::kSb + swz(g + 8, nt, 128) + 4 * tg) = pack_bf16(cs[2], cs[3]);
    }
  };
  // Z of tile v: the sum of the four quarter partials, for the rows inside the sequence.
  auto z_sum = [&](int v) {
    const int t = tid >> 5, j = (tid & 31) * 2;
    float2 z = make_float2(0.f, 0.f);
#pragma unroll
    for (int kq = 0; kq < 4; ++kq) {
      const float2 x = *reinterpret_cast<const float2*>(partZ + kq * kTile * kPad + t * kPad + j);
      z.x += x.x;
      z.y += x.y;
    }
    const int tt = v * kTile + t;
    if (tt < p.T) {
      __nv_bfloat16* Z = static_cast<__nv_bfloat16*>(p.Z) + (static_cast<size_t>(unit) * p.T + tt) * kD + j;
      *reinterpret_cast<uint32_t*>(Z) = pack_bf16(z.x, z.y);
    }
  };

  bool ok = true;
  if (n_tiles > 0) {
    ok = wait_tile(0);
    if (!__syncthreads_or(!ok)) {
      phase_u(0);
      __syncthreads();
    } else {
      ok = false;
    }
  }
  for (int u = 0; ok && u < n_tiles; ++u) {
    const int s = u & 1;
    const uint32_t sQ = s0 + pipe::kQKV + s * 3 * kTileBytes, sK = sQ + kTileBytes;
    const uint8_t* sVp = sm + pipe::kQKV + s * 3 * kTileBytes + 2 * kTileBytes;
    const uint32_t Acur = s0 + pipe::kAb + s * pipe::kABytes;
    const uint32_t W2cur = s0 + pipe::kW2b + s * pipe::kW2Bytes;
    uint8_t* W2next = sm + pipe::kW2b + (s ^ 1) * pipe::kW2Bytes;

    // (G) G partials of tile u: warp -> value columns [16(w&3), +16), hidden quarter w>>2;
    //     and the Z of tile u - 1.
    {
      const int np = warp & 3, kq = warp >> 2;
      float cg[2][4] = {};
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        uint32_t a[4], b[4];
        ldA(a, Acur, kRowM, 0, 8 * kq + 2 * ks, lane);
        ldBT(b, W2cur, 128, 64 * kq + 16 * ks, 2 * np, lane);
        mma2(cg, a, b);
      }
      float* dst = partG + kq * kTile * kPad;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int c = 16 * np + 8 * nt + 2 * tg;
        *reinterpret_cast<float2*>(dst + g * kPad + c) = make_float2(cg[nt][0], cg[nt][1]);
        *reinterpret_cast<float2*>(dst + (g + 8) * kPad + c) = make_float2(cg[nt][2], cg[nt][3]);
      }
    }
    if (u > 0) z_sum(u - 1);
    __syncthreads();
    // (R) G = sum of the quarters - V, bf16.
    {
      const int t = tid >> 5, j = (tid & 31) * 2;
      float2 acc = make_float2(0.f, 0.f);
#pragma unroll
      for (int kq = 0; kq < 4; ++kq) {
        const float2 v = *reinterpret_cast<const float2*>(partG + kq * kTile * kPad + t * kPad + j);
        acc.x += v.x;
        acc.y += v.y;
      }
      const uint32_t vv = *reinterpret_cast<const uint32_t*>(sVp + swz(t, j >> 3, 128) + (j & 7) * 2);
      acc.x -= bf16_lo(vv);
      acc.y -= bf16_hi(vv);
      *reinterpret_cast<uint32_t*>(sm + pipe::kGb + swz(t, j >> 3, 128) + (j & 7) * 2) = pack_bf16(acc.x, acc.y);
    }
    __syncthreads();

    // (DH) D = (G W2^T) .* P and the W2 update; Hq, Aq and the W1 update (this warp's hidden units).
    uint32_t bd[4];
    {
      float cd[2][4] = {};
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        uint32_t a[4], b[4];
        ldA(a, Gb, 128, 0, 2 * ks, lane);
        ldB(b, W2cur, 128, 16 * warp, 2 * ks, lane);
        mma2(cd, a, b);
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) cd[nt][r] *= cp[nt][r];
      bd[0] = movm_t(pack_bf16(cd[0][0], cd[0][1]));
      bd[1] = movm_t(pack_bf16(cd[0][2], cd[0][3]));
      bd[2] = movm_t(pack_bf16(cd[1][0], cd[1][1]));
      bd[3] = movm_t(pack_bf16(cd[1][2], cd[1][3]));
      uint32_t a[4];
      ldAT(a, Acur, kRowM, 0, 2 * warp, lane);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t b[4];
        ldBT(b, Gb, 128, 0, 2 * q, lane);
        float acc[2][4] = {};
        mma2(acc, a, b);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int r = 0; r < 4; ++r) w2[2 * q + nt][r] = fmaf(-eta, acc[nt][r], w2[2 * q + nt][r]);
      }
    }
    {
      float ch[2][4] = {}, cs[2][4] = {};
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        uint32_t a[4], b[4];
        ldA(a, sQ, 128, 0, 2 * ks, lane);
        ldBT(b, W1b, kRowM, 16 * ks, 2 * warp, lane);
        mma2(ch, a, b);
      }
      {
        uint32_t a[4];
        ldA(a, Sb, 128, 0, 0, lane);
        mma2(cs, a, bd);
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) ch[nt][r] = gelu1(fmaf(-eta, cs[nt][r], ch[nt][r]));
      st_tile(sm + pipe::kAqb, kRowM, 0, warp, ch, lane);
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        uint32_t a[4];
        ldAT(a, sK, 128, 0, 2 * mt, lane);
        float acc[2][4] = {};
        mma2(acc, a, bd);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int r = 0; r < 4; ++r) w1[mt][nt][r] = fmaf(-eta, acc[nt][r], w1[mt][nt][r]);
      }
    }
    // Columns [16w, +16) of the W1 copy are read by this warp alone: rewrite them now.
    __syncwarp();
    TTT_STORE_W1(sm + pipe::kW1b);
    // Tile u's stage has been read for the last time (the proxy fence orders those reads
    // before the refill's async-proxy write); tile u + 1 must have landed.
    const bool mine = u + 1 < n_tiles ? wait_tile(u + 1) : true;
    fence_proxy_async_smem();
    if (__syncthreads_or(!mine)) {
      ok = false;
      break;
    }
    if (tid == 0 && u + 2 < n_tiles) load_tile(u + 2);

    // (N) U, A, P, tril(QK^T) of tile u + 1; Z partials of tile u; tile u's new W2 into the other copy.
    if (u + 1 < n_tiles) phase_u(u + 1);
    {
      const int np = warp & 3, kq = warp >> 2;
      float cz[2][4] = {}, csa[2][4] = {};
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        uint32_t a[4], b[4], ba[4];
        ldA(a, Aqb, kRowM, 0, 8 * kq + 2 * ks, lane);
        ldBT(b, W2cur, 128, 64 * kq + 16 * ks, 2 * np, lane);
        ldB(ba, Acur, kRowM, 0, 8 * kq + 2 * ks, lane);
        mma2(cz, a, b);
        mma2(csa, a, ba);
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {  // keep t2 <= t, scale by -eta
        const int c = 8 * nt + 2 * tg;
        csa[nt][0] = c > g ? 0.f : -eta * csa[nt][0];
        csa[nt][1] = c + 1 > g ? 0.f : -eta * csa[nt][1];
        csa[nt][2] = c > g + 8 ? 0.f : -eta * csa[nt][2];
        csa[nt][3] = c + 1 > g + 8 ? 0.f : -eta * csa[nt][3];
      }
      const uint32_t sa[4] = {pack_bf16(csa[0][0], csa[0][1]), pack_bf16(csa[0][2], csa[0][3]),
                              pack_bf16(csa[1][0], csa[1][1]), pack_bf16(csa[1][2], csa[1][3])};
      uint32_t bg[4];
      ldBT(bg, Gb, 128, 0, 2 * np, lane);
      mma2(cz, sa, bg);
      float* dst = partZ + kq * kTile * kPad;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int c = 16 * np + 8 * nt + 2 * tg;
        *reinterpret_cast<float2*>(dst + g * kPad + c) = make_float2(cz[nt][0], cz[nt][1]);
        *reinterpret_cast<float2*>(dst + (g + 8) * kPad + c) = make_float2(cz[nt][2], cz[nt][3]);
      }
    }
    TTT_STORE_W2(W2next);
    __syncthreads();
  }
  if (ok && n_tiles > 0) z_sum(n_tiles - 1);
  // Loads still in flight when a wait gave up must land before the CTA exits.
  if (!ok && tid == 0)
    for (int v = issued > 2 ? issued - 2 : 0; v < issued; ++v)
      (void)mbar_wait_bounded(&full[v & 1], (v >> 1) & 1, p.timeout_ns);
  // Final state.
  float* W1o = p.W1_out + static_cast<size_t>(unit) * kD * kM;
  float* W2o = p.W2_out + static_cast<size_t>(unit) * kM * kD;
#pragma unroll
  for (int mt = 0; mt < 4; ++mt)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int i = 16 * mt + g, c = 16 * warp + 8 * nt + 2 * tg;
      *reinterpret_cast<float2*>(W1o + i * kM + c) = make_float2(w1[mt][nt][0], w1[mt][nt][1]);
      *reinterpret_cast<float2*>(W1o + (i + 8) * kM + c) = make_float2(w1[mt][nt][2], w1[mt][nt][3]);
    }
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    const int r = 16 * warp + g, c = 8 * nt + 2 * tg;
    *reinterpret_cast<float2*>(W2o + r * kD + c) = make_float2(w2[nt][0], w2[nt][1]);
    *reinterpret_cast<float2*>(W2o + (r + 8) * kD + c) = make_float2(w2[nt][2], w2[nt][3]);
  }
}

#undef TTT_STORE_W1
#undef TTT_STORE_W2

}  // namespace

bool mlp_mma_supported(const MlpParams& p) { return p.bf16 && p.d == kD && p.m == kM && p.b % kTile == 0; }

int mlp_mma_tile_rows() { return kTile; }

cudaError_t launch_mlp_mma(const MlpParams& p, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                           cudaStream_t stream) {
  if (p.units == 0) return cudaSuccess;
  if (p.b == kTile) {
    const int smem = pipe::kBytes + 1024;
    const cudaError_t e = cudaFuncSetAttribute(mlp_mma16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    mlp_mma16_kernel<<<p.units, kThreads, smem, stream>>>(mq, mk, mv, p);
    return cudaGetLastError();
  }
  const int smem = kBaseBytes + (p.b > kTile ? kSnapBytes : 0) + 1024;
  const cudaError_t e = cudaFuncSetAttribute(mlp_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  mlp_mma_kernel<<<p.units, kThreads, smem, stream>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace ttt
