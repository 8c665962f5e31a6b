// TTT-MLP forward for b = 16 on a cluster of two CTAs per (batch row, head):
// each CTA owns half of the 256 hidden units, so a unit's work spreads over two
// SMs (96 of 148 SMs for B4 H12 instead of 48).
//
// Method as mlp_mma.cu ("Test-Time Training (TTT) guide", section 3: two layers,
// hidden 4x, GELU; "5 · TestingTime 训练与长上下文", section 1.1: gradients at the
// chunk-start weights, dual form). Per 16-token tile (b = 16: every tile is a chunk):
//   U = K W1, A = gelu(U), P = gelu'(U)              (own hidden units)
//   G = A W2 - V                                     (a sum over all hidden units)
//   D = (G W2^T) .* P, Hq = Q W1 - eta tril(Q K^T) D, Aq = gelu(Hq)   (own)
//   W2 -= eta A^T G, W1 -= eta K^T D                 (own rows / columns)
//   Z = Aq W2 - eta tril(Aq A^T) G                   (a sum over all hidden units)
// Everything but the two sums is local to the hidden units, so only G and Z cross
// between the CTAs. Each CTA splits its 128 hidden units into two quarters of 64;
// a warp forms the 16 x 16 block of a quarter's partial G (or Z) for 16 value
// columns and writes it to both CTAs' shared memory: locally with plain stores,
// to the peer with st.async, whose bytes complete a transaction count on the
// peer's mbarrier. So both CTAs hold all four quarters of G; Z's blocks go to the
// CTA that writes those 32 columns of Z. The exchange buffers are double-buffered
// by tile parity and every mbarrier wait is bounded. Each mbarrier phase is armed
// (expect_tx) two tiles ahead, after the buffer's last read, which always precedes
// the peer's next send into it (the peer's send of tile u + 2 needs this CTA's
// partial of tile u + 2). A cluster barrier at the start (the peer's barriers are
// initialised and armed) and at the end (no st.async still targets an exited CTA)
// are the only unbounded waits; both CTAs always reach both.
#include "kernels.h"
#include "mlp_frag.cuh"
#include "ttt_device.cuh"

namespace ttt {
namespace {

using namespace mlpf;

constexpr int kD = 64;
constexpr int kM = 256;                 // hidden units of a unit
constexpr int kMh = 128;                // ... of one CTA
constexpr int kTile = 16;
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kTileBytes = kTile * kD * 2;
constexpr int kRowH = kMh * 2;          // 256-byte rows of [.][128] bf16
constexpr int kPad = 68;                // fp32 row stride of the G partials
constexpr int kPadZ = 36;               // ... of the Z partials (32 columns)
// shared memory map (bytes from a 1024-aligned base)
constexpr int kQKV = 0;                                  // [2 stages][Q, K, V]
constexpr int kW1b = kQKV + 2 * 3 * kTileBytes;          // W1[:, own], bf16 [64][128]
constexpr int kW2b = kW1b + kD * kRowH;                  // W2[own, :], bf16 [128][64]
constexpr int kAb = kW2b + kMh * 128;                    // A, bf16 [16][128]
constexpr int kAqb = kAb + kTile * kRowH;                // Aq, bf16 [16][128]
constexpr int kGb = kAqb + kTile * kRowH;                // G, bf16 [16][64]
constexpr int kSb = kGb + kTile * 128;                   // tril(Q K^T), bf16 [16][16] in 128-byte rows
constexpr int kPartG = kSb + kTile * 128;                // [2 parity][4 quarters][16][kPad] fp32
constexpr int kPartGBytes = 4 * kTile * kPad * 4;
constexpr int kPartZ = kPartG + 2 * kPartGBytes;         // [2 parity][4 quarters][16][kPadZ] fp32
constexpr int kPartZBytes = 4 * kTile * kPadZ * 4;
constexpr int kBar = kPartZ + 2 * kPartZBytes;           // full[2], gfull[2], zfull[2]
constexpr int kSmemBytes = kBar + 64 + 1024;
static_assert(kSmemBytes <= 227 * 1024, "fits one CTA per SM");
constexpr uint32_t kGRecv = 8 * kTile * 16 * 4;          // the peer's 8 warps: a 16 x 16 fp32 block each
constexpr uint32_t kZRecv = 4 * kTile * 16 * 4;          // 4 of the peer's warps serve this CTA's columns

enum : int { kWhereClLoad = 40, kWhereClG = 41, kWhereClZ = 42 };

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t map_peer(uint32_t addr, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(addr), "r"(rank));
  return d;
}
// Eight bytes into the peer's shared memory; their arrival completes 8 bytes of the
// transaction count of the peer's mbarrier.
__device__ __forceinline__ void st_async_f2(uint32_t remote, float a, float b, uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(remote),
               "f"(a), "f"(b), "r"(remote_bar)
               : "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    mlp_cluster_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                       const __grid_constant__ CUtensorMap mv, MlpParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + kBar);  // [2] TMA
  uint64_t* gfull = full + 2;                                // [2] the peer's G blocks of a tile parity
  uint64_t* zfull = full + 4;                                // [2] the peer's Z blocks
  const uint32_t s0 = smem_u32(sm);
  float* partG = reinterpret_cast<float*>(sm + kPartG);
  float* partZ = reinterpret_cast<float*>(sm + kPartZ);

  const uint32_t rank = cluster_rank();
  const uint32_t peer = rank ^ 1u;
  const int unit = blockIdx.x >> 1;
  const int h = unit % p.H;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, tg = lane & 3;
  const int hid = static_cast<int>(rank) * kMh + 16 * warp;  // this warp's first hidden unit (of 256)
  const float eta = p.eta[h];
  const int n_tiles = (p.T + kTile - 1) / kTile;

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&gfull[i], 1);
      mbar_init(&zfull[i], 1);
    }
    fence_barrier_init();
    // Arm the exchange barriers for tiles 0 and 1 (later tiles: after each buffer's last read).
    for (int v = 0; v < 2 && v < n_tiles; ++v) {
      mbar_arrive_expect_tx(&gfull[v], kGRecv);
      mbar_arrive_expect_tx(&zfull[v], kZRecv);
    }
  }
  // fp32 masters: W1[:, hid:hid+16] (C fragments, 4 m-tiles x 2 n-tiles) and W2[hid:hid+16, :].
  float w1[4][2][4], w2[8][4];
  {
    const float* W10 = p.W1_0 + static_cast<size_t>(h) * kD * kM;
    const float* W20 = p.W2_0 + static_cast<size_t>(h) * kM * kD;
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int i = 16 * mt + g, c = hid + 8 * nt + 2 * tg;
        w1[mt][nt][0] = W10[i * kM + c];
        w1[mt][nt][1] = W10[i * kM + c + 1];
        w1[mt][nt][2] = W10[(i + 8) * kM + c];
        w1[mt][nt][3] = W10[(i + 8) * kM + c + 1];
      }
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int r = hid + g, c = 8 * nt + 2 * tg;
      w2[nt][0] = W20[r * kD + c];
      w2[nt][1] = W20[r * kD + c + 1];
      w2[nt][2] = W20[(r + 8) * kD + c];
      w2[nt][3] = W20[(r + 8) * kD + c + 1];
    }
  }
  // bf16 copies of this warp's slices (local hidden index 16 * warp).
  auto store_w1 = [&]() {
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int ch = 2 * warp + nt;
        *reinterpret_cast<uint32_t*>(sm + kW1b + swz(16 * mt + g, ch, kRowH) + 4 * tg) =
            pack_bf16(w1[mt][nt][0], w1[mt][nt][1]);
        *reinterpret_cast<uint32_t*>(sm + kW1b + swz(16 * mt + g + 8, ch, kRowH) + 4 * tg) =
            pack_bf16(w1[mt][nt][2], w1[mt][nt][3]);
      }
  };
  auto store_w2 = [&]() {
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      *reinterpret_cast<uint32_t*>(sm + kW2b + swz(16 * warp + g, nt, 128) + 4 * tg) = pack_bf16(w2[nt][0], w2[nt][1]);
      *reinterpret_cast<uint32_t*>(sm + kW2b + swz(16 * warp + g + 8, nt, 128) + 4 * tg) =
          pack_bf16(w2[nt][2], w2[nt][3]);
    }
  };
  store_w1();
  store_w2();
  __syncthreads();
  cluster_sync();  // the peer's barriers are initialised and armed before anything is sent to it

  int issued = 0;
  auto load_tile = [&](int u) {
    const int s = u & 1;
    uint8_t* st = sm + kQKV + s * 3 * kTileBytes;
    mbar_arrive_expect_tx(&full[s], 3 * kTileBytes);
    tma_load_3d(st, &mq, &full[s], 0, u * kTile, unit);
    tma_load_3d(st + kTileBytes, &mk, &full[s], 0, u * kTile, unit);
    tma_load_3d(st + 2 * kTileBytes, &mv, &full[s], 0, u * kTile, unit);
    issued = u + 1;
  };
  if (tid == 0 && n_tiles > 0) {
    prefetch_tmap(&mq);
    prefetch_tmap(&mk);
    prefetch_tmap(&mv);
    load_tile(0);
  }

  const uint32_t W1b = s0 + kW1b, W2b = s0 + kW2b, Ab = s0 + kAb, Aqb = s0 + kAqb, Gb = s0 + kGb, Sb = s0 + kSb;
  const uint32_t gbar_peer[2] = {map_peer(smem_u32(&gfull[0]), peer), map_peer(smem_u32(&gfull[1]), peer)};
  const uint32_t zbar_peer[2] = {map_peer(smem_u32(&zfull[0]), peer), map_peer(smem_u32(&zfull[1]), peer)};
  bool ok = true;
  bool late_fail = false;        // a wait of the previous tile's Z phase gave up
  for (int u = 0; ok && u < n_tiles; ++u) {
    const int s = u & 1;
    const uint32_t ph = static_cast<uint32_t>(u >> 1) & 1u;
    const uint32_t sQ = s0 + kQKV + s * 3 * kTileBytes, sK = sQ + kTileBytes;
    const uint8_t* sVp = sm + kQKV + s * 3 * kTileBytes + 2 * kTileBytes;
    float* pg = partG + s * (kPartGBytes / 4);
    float* pz = partZ + s * (kPartZBytes / 4);

    // Tile start: its data has landed; the stage of tile u - 1 and every buffer of the
    // previous tile are free.
    bool mine = mbar_wait_bounded(&full[s], ph, p.timeout_ns);
    if (!mine) report_error(p.status, TTT_ERR_TIMEOUT, kWhereClLoad, unit);
    fence_proxy_async_smem();
    if (__syncthreads_or(!mine || late_fail)) {
      ok = false;
      break;
    }
    if (tid == 0) {
      if (u + 1 < n_tiles) load_tile(u + 1);
      // Z blocks of tile u - 1 are read (all threads passed the barrier above): arm for tile u + 1.
      if (u >= 1 && u + 1 < n_tiles) mbar_arrive_expect_tx(&zfull[s ^ 1], kZRecv);
    }

    // (1) U = K W1, A = gelu(U), P = gelu'(U) for this warp's hidden units; warps 0 and 1
    //     form one n-tile each of tril(Q K^T).
    float cp[2][4];
    {
      float cu[2][4] = {};
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        uint32_t a[4], b[4];
        ldA(a, sK, 128, 0, 2 * ks, lane);
        ldBT(b, W1b, kRowH, 16 * ks, 2 * warp, lane);
        mma2(cu, a, b);
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) gelu2(cu[nt][r], cu[nt][r], cp[nt][r]);
      st_tile(sm + kAb, kRowH, 0, warp, cu, lane);
      if (warp < 2) {
        const int nt = warp;
        float cs[4] = {};
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          uint32_t a[4], b[4];
          ldA(a, sQ, 128, 0, 2 * ks, lane);
          ldB(b, sK, 128, 0, 2 * ks, lane);
          const uint32_t bn[2] = {b[2 * nt], b[2 * nt + 1]};
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
    }
    __syncthreads();

    // (2) This CTA's quarter kq = w >> 2 of G for value columns [16 np, +16), np = w & 3,
    //     into quarter slot 2 rank + kq of both CTAs.
    {
      const int np = warp & 3, kq = warp >> 2;
      float cg[2][4] = {};
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        uint32_t a[4], b[4];
        ldA(a, Ab, kRowH, 0, 8 * kq + 2 * ks, lane);
        ldBT(b, W2b, 128, 64 * kq + 16 * ks, 2 * np, lane);
        mma2(cg, a, b);
      }
      float* dst = pg + (2 * static_cast<int>(rank) + kq) * kTile * kPad;
      const uint32_t rdst = map_peer(smem_u32(dst), peer);
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int c = 16 * np + 8 * nt + 2 * tg;
        *reinterpret_cast<float2*>(dst + g * kPad + c) = make_float2(cg[nt][0], cg[nt][1]);
        *reinterpret_cast<float2*>(dst + (g + 8) * kPad + c) = make_float2(cg[nt][2], cg[nt][3]);
        st_async_f2(rdst + (g * kPad + c) * 4, cg[nt][0], cg[nt][1], gbar_peer[s]);
        st_async_f2(rdst + ((g + 8) * kPad + c) * 4, cg[nt][2], cg[nt][3], gbar_peer[s]);
      }
    }
    // The peer's two quarters (bounded wait on their bytes) and this CTA's (the barrier).
    mine = mbar_wait_bounded(&gfull[s], ph, p.timeout_ns);
    if (!mine) report_error(p.status, TTT_ERR_TIMEOUT, kWhereClG, unit);
    if (__syncthreads_or(!mine)) {
      ok = false;
      break;
    }

    // (3) G = the sum of the four quarters - V, bf16 (four columns per thread).
    {
      const int t = tid >> 4, j = (tid & 15) * 4;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 v = *reinterpret_cast<const float4*>(pg + q * kTile * kPad + t * kPad + j);
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
      const uint2 vv = *reinterpret_cast<const uint2*>(sVp + swz(t, j >> 3, 128) + (j & 7) * 2);
      *reinterpret_cast<uint2*>(sm + kGb + swz(t, j >> 3, 128) + (j & 7) * 2) =
          make_uint2(pack_bf16(acc.x - bf16_lo(vv.x), acc.y - bf16_hi(vv.x)),
                     pack_bf16(acc.z - bf16_lo(vv.y), acc.w - bf16_hi(vv.y)));
    }
    __syncthreads();
    // The G slots of this parity are read: arm them for tile u + 2.
    if (tid == 0 && u + 2 < n_tiles) mbar_arrive_expect_tx(&gfull[s], kGRecv);

    // (4) D = (G W2^T) .* P and the W2 update; Hq, Aq and the W1 update (this warp's hidden units).
    uint32_t bd[4];
    {
      float cd[2][4] = {};
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        uint32_t a[4], b[4];
        ldA(a, Gb, 128, 0, 2 * ks, lane);
        ldB(b, W2b, 128, 16 * warp, 2 * ks, lane);
        mma2(cd, a, b);
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) cd[nt][r] *= cp[nt][r];
      // D as the B operand (k = t, n = hidden) of S D and K^T D, by transposing its 8 x 8 blocks.
      bd[0] = movm_t(pack_bf16(cd[0][0], cd[0][1]));
      bd[1] = movm_t(pack_bf16(cd[0][2], cd[0][3]));
      bd[2] = movm_t(pack_bf16(cd[1][0], cd[1][1]));
      bd[3] = movm_t(pack_bf16(cd[1][2], cd[1][3]));
      uint32_t a[4];
      ldAT(a, Ab, kRowH, 0, 2 * warp, lane);
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
        ldBT(b, W1b, kRowH, 16 * ks, 2 * warp, lane);
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
      st_tile(sm + kAqb, kRowH, 0, warp, ch, lane);
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
    // This warp's columns of the W1 copy are read by this warp alone: rewrite them now.
    __syncwarp();
    store_w1();
    __syncthreads();  // Aq complete

    // (5) Quarter kq's block of Z for value columns [16 np, +16) (with its block of
    //     tril(Aq A^T) applied to G), to the CTA that writes those columns: np < 2 rank 0.
    {
      const int np = warp & 3, kq = warp >> 2;
      float cz[2][4] = {}, csa[2][4] = {};
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        uint32_t a[4], b[4], ba[4];
        ldA(a, Aqb, kRowH, 0, 8 * kq + 2 * ks, lane);
        ldBT(b, W2b, 128, 64 * kq + 16 * ks, 2 * np, lane);
        ldB(ba, Ab, kRowH, 0, 8 * kq + 2 * ks, lane);
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
      float* dst = pz + (2 * static_cast<int>(rank) + kq) * kTile * kPadZ;
      const bool local = static_cast<uint32_t>(np >> 1) == rank;
      const uint32_t rdst = map_peer(smem_u32(dst), peer);
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int c = 16 * (np & 1) + 8 * nt + 2 * tg;
        if (local) {
          *reinterpret_cast<float2*>(dst + g * kPadZ + c) = make_float2(cz[nt][0], cz[nt][1]);
          *reinterpret_cast<float2*>(dst + (g + 8) * kPadZ + c) = make_float2(cz[nt][2], cz[nt][3]);
        } else {
          st_async_f2(rdst + (g * kPadZ + c) * 4, cz[nt][0], cz[nt][1], zbar_peer[s]);
          st_async_f2(rdst + ((g + 8) * kPadZ + c) * 4, cz[nt][2], cz[nt][3], zbar_peer[s]);
        }
      }
    }
    __syncthreads();  // every read of this tile's W2, A, Aq and G copies is done; our Z blocks are written
    store_w2();       // this warp's rows of the updated W2

    // Z of this CTA's 32 columns: the peer's blocks (bounded wait) and ours.
    mine = mbar_wait_bounded(&zfull[s], ph, p.timeout_ns);
    if (!mine) {
      report_error(p.status, TTT_ERR_TIMEOUT, kWhereClZ, unit);
      late_fail = true;
    } else {
      const int t = tid >> 4, j = (tid & 15) * 2;
      float2 z = make_float2(0.f, 0.f);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 v = *reinterpret_cast<const float2*>(pz + q * kTile * kPadZ + t * kPadZ + j);
        z.x += v.x;
        z.y += v.y;
      }
      const int tt = u * kTile + t;
      if (tt < p.T) {
        __nv_bfloat16* Z = static_cast<__nv_bfloat16*>(p.Z) + (static_cast<size_t>(unit) * p.T + tt) * kD +
                           32 * static_cast<int>(rank) + j;
        *reinterpret_cast<uint32_t*>(Z) = pack_bf16(z.x, z.y);
      }
    }
  }
  if (late_fail) ok = false;
  // TMA loads still in flight when a wait gave up must land before the CTA exits.
  if (!ok && tid == 0)
    for (int v = issued > 2 ? issued - 2 : 0; v < issued; ++v)
      (void)mbar_wait_bounded(&full[v & 1], (v >> 1) & 1, p.timeout_ns);

  // Final state: this CTA's columns of W1 and rows of W2.
  float* W1o = p.W1_out + static_cast<size_t>(unit) * kD * kM;
  float* W2o = p.W2_out + static_cast<size_t>(unit) * kM * kD;
#pragma unroll
  for (int mt = 0; mt < 4; ++mt)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int i = 16 * mt + g, c = hid + 8 * nt + 2 * tg;
      *reinterpret_cast<float2*>(W1o + i * kM + c) = make_float2(w1[mt][nt][0], w1[mt][nt][1]);
      *reinterpret_cast<float2*>(W1o + (i + 8) * kM + c) = make_float2(w1[mt][nt][2], w1[mt][nt][3]);
    }
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    const int r = hid + g, c = 8 * nt + 2 * tg;
    *reinterpret_cast<float2*>(W2o + r * kD + c) = make_float2(w2[nt][0], w2[nt][1]);
    *reinterpret_cast<float2*>(W2o + (r + 8) * kD + c) = make_float2(w2[nt][2], w2[nt][3]);
  }
  cluster_sync();  // the peer sends nothing more into this CTA's shared memory
}

}  // namespace

bool mlp_cluster_supported(const MlpParams& p) { return p.bf16 && p.d == kD && p.m == kM && p.b == kTile; }

cudaError_t launch_mlp_cluster(const MlpParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                               const CUtensorMap& mv, cudaStream_t stream) {
  if (p.units == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(mlp_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * p.units);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, mlp_cluster_kernel, mq, mk, mv, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace ttt
