// Backward of the chunked TTT-Linear scan on the tensor cores: bf16 Q, K, V,
// dZ (dQ, dK, dV written in bf16), fp32 state and accumulation, d = 64, b = 16.
//
// The outer loop trains W0, eta and the projections that make Q, K, V by
// backpropagating through the inner loop ("5 · TestingTime 训练与长上下文",
// section 2.2). For chunk c with start state W and G the gradient of the next
// chunk's start state (G = dW_out after the last chunk):
//   E = K W - V,  S = tril(Q K^T),  P = -eta tril(dZ E^T)
//   dE = -eta (K G + S^T dZ),  dV = -dE
//   dQ = dZ W^T + P K,  dK = -eta E G^T + P^T Q + dE W^T
//   d eta += -sum(E .* K G) - sum(S .* dZ E^T)
//   G <- G + Q^T dZ + K^T dE,   and dW0 = G after the first chunk
// (the same recurrence as linear_bwd.cu, which serves fp32 and other shapes).
//
// Design. The chunk rule splits over the output columns j of W, and so do E, G
// and dE: each of 4 consumer warps owns 16 columns and keeps G^T (16 x 64) as
// fp32 mma.sync accumulator fragments for the whole sequence. dQ, dK and P sum
// over all columns: once every warp has written its columns of G and dE (bf16,
// shared memory), each warp forms the full P and the dQ, dK of its own band of
// 16 input features from those full-width copies, so a chunk needs one meeting
// of the four warps. The copies of W, E (per block) and of G, dE (per chunk)
// are kept twice, so that the next one can be written while the last is read.
//   Pass 1 walks the sequence forward (K, V only), keeping W in fragments as the
//   forward kernel does, and writes W at the start of every 64-token block to
//   the workspace (fp32).
//   Pass 2 walks the blocks in reverse. For a block it reloads W, recomputes the
//   four chunk states and errors (bf16 copies in shared memory), then runs the
//   backward of its four chunks, last first.
// A producer warp streams the 64-token blocks by TMA (K, V for pass 1; Q, K, V,
// dZ for pass 2, double-buffered) and forms, per chunk, S = tril(Q K^T) and
// S^T = triu(K Q^T) as the consumers' B fragments. Every wait is bounded in
// wall-clock time; a role that gives up sets a shared flag the others see.
#include "ttt_device.cuh"
#include "kernels.h"

namespace ttt {
namespace {

constexpr int kD = 64;
constexpr int kTile = 16;               // = b
constexpr int kBlk = 64;                // tokens per block (4 chunks)
constexpr int kWarps = 4;               // consumer warps; one more produces
constexpr int kThreads = (kWarps + 1) * 32;
constexpr int kTileBytes = kTile * kD * 2;   // 2 KB
constexpr int kBlkBytes = kBlk * kD * 2;     // 8 KB
// shared memory map (bytes from a 1024-aligned base)
constexpr int kP1 = 0;                                  // pass 1: [2 stages][K, V] blocks
constexpr int kP2 = kP1 + 2 * 2 * kBlkBytes;            // pass 2: [2 stages][Q, K, V, dZ] blocks
constexpr int kSb = kP2 + 2 * 4 * kBlkBytes;            // [2 stages][4 chunks][S, S^T] B fragments, 512 B each
constexpr int kWcBytes = 4 * kD * kD * 2;             // [4 chunks] W bf16 [i][j]
constexpr int kEcBytes = 4 * kTileBytes;                // [4 chunks] E bf16 [t][j]
constexpr int kWc = kSb + 2 * 4 * 2 * 512;              // [2 blocks] W copies
constexpr int kEc = kWc + 2 * kWcBytes;                 // [2 blocks] E copies
constexpr int kGc = kEc + 2 * kEcBytes;                 // [2 chunks] G bf16 [i][j]
constexpr int kDE = kGc + 2 * kD * kD * 2;              // [2 chunks] dE bf16 [t][j]
constexpr int kOut = kDE + 2 * kTileBytes;              // [4 warps][2] 16 x 16 bf16 output staging
constexpr int kRed = kOut + kWarps * 2 * 512;           // d eta per warp
constexpr int kBar = kRed + 64;
constexpr int kNumBars = 11;
constexpr int kMisc = kBar + kNumBars * 8;              // abort flag
constexpr int kSmemBytes = kMisc + 16 + 1024;
static_assert(kSmemBytes <= 227 * 1024, "fits one CTA per SM");

enum : int { kWhereBwdProducer = 20, kWhereBwdPass1 = 21, kWhereBwdPass2 = 22, kWhereBwdSync = 23 };

__device__ __forceinline__ void unpack4(uint4 v, float (&s)[2][4]) {
  // the producer packs C fragments as {(nt0: r0, r1), (nt1: r0, r1), (nt0: r2, r3), (nt1: r2, r3)}
  s[0][0] = bf16_lo(v.x); s[0][1] = bf16_hi(v.x);
  s[1][0] = bf16_lo(v.y); s[1][1] = bf16_hi(v.y);
  s[0][2] = bf16_lo(v.z); s[0][3] = bf16_hi(v.z);
  s[1][2] = bf16_lo(v.w); s[1][3] = bf16_hi(v.w);
}

// A fragments (bf16) of a 16 x 64 block of X^T held as fp32 C fragments xt[8][4]
// (rows m, columns 8q + 2tg): k-step s covers columns [16s, 16s + 16).
__device__ __forceinline__ void pack_a(const float (&xt)[8][4], uint32_t (&a)[4][4]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    a[k][0] = pack_bf16(xt[2 * k][0], xt[2 * k][1]);
    a[k][1] = pack_bf16(xt[2 * k][2], xt[2 * k][3]);
    a[k][2] = pack_bf16(xt[2 * k + 1][0], xt[2 * k + 1][1]);
    a[k][3] = pack_bf16(xt[2 * k + 1][2], xt[2 * k + 1][3]);
  }
}

// Writes X (64 x 64, [i][j], 128-byte swizzled rows) columns [16w, 16w + 16) from
// the A fragments of X^T rows j (a transposing stmatrix per 16 x 16 block).
__device__ __forceinline__ void store_t(uint32_t base, const uint32_t (&a)[4][4], int warp, int lane) {
  const int mi = lane >> 3, mr = lane & 7;
#pragma unroll
  for (int s = 0; s < 4; ++s) stsm_x4_t(base + swz128(16 * s + ((mi >> 1) << 3) + mr, 2 * warp + (mi & 1)), a[s]);
}

// kSeg: the unit's sequence is cut into p.bseg_count segments (one CTA each);
// without it every CTA takes a whole unit.
template <bool kSeg>
__global__ void __launch_bounds__(kThreads, 1)
    linear_bwd_mma_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                          const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdz,
                          LinearBwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full1 = reinterpret_cast<uint64_t*>(sm + kBar);
  uint64_t* empty1 = full1 + 2;
  uint64_t* full2 = full1 + 4;
  uint64_t* ready2 = full1 + 6;
  uint64_t* empty2 = full1 + 8;
  uint64_t* sync1 = full1 + 10;  // the four consumer warps meet (copies of W, E, G, dE written)
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kMisc);
  const uint32_t s0 = smem_u32(sm);

  // One CTA per (unit, segment): blocks [blk0, blk1) of 64 tokens (all of them without segments).
  const int S = kSeg ? p.bseg_count : 1;
  const int unit = blockIdx.x / S;
  const int seg = blockIdx.x % S;
  const int h = unit % p.H;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tg = lane & 3, mi = lane >> 3, mr = lane & 7;
  const int T = p.T;
  const int ntiles = (T + kTile - 1) / kTile;
  const int nblk_all = (T + kBlk - 1) / kBlk;
  const int blk0 = kSeg ? seg * (p.bseg_len / kBlk) : 0;
  const int blk1 = kSeg ? min(nblk_all, blk0 + p.bseg_len / kBlk) : nblk_all;
  const int nblk = blk1 - blk0;  // this CTA's blocks
  const float eta = p.eta[h];

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&full1[i], 1);
      mbar_init(&empty1[i], kWarps);
      mbar_init(&full2[i], 1);
      mbar_init(&ready2[i], 1);
      mbar_init(&empty2[i], kWarps);
    }
    mbar_init(sync1, kWarps);
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kWarps) {
    // ---------------------------------------------------------------- producer
    bool ok = true;
    int issued1 = 0, issued2 = 0, seen2 = 0;  // lane 0's TMA blocks, and those seen to land
    if (lane == 0) {
      prefetch_tmap(&mk);
      prefetch_tmap(&mv);
      prefetch_tmap(&mq);
      prefetch_tmap(&mdz);
      for (int lb = 0; lb < nblk && ok; ++lb) {
        const int s = lb & 1, bk = blk0 + lb;
        if (lb >= 2) ok = mbar_wait_or_abort(&empty1[s], ((lb >> 1) - 1) & 1, p.timeout_ns, abort_flag);
        if (!ok) break;
        mbar_arrive_expect_tx(&full1[s], 2 * kBlkBytes);
        tma_load_3d(sm + kP1 + s * 2 * kBlkBytes, &mk, &full1[s], 0, bk * kBlk, unit);
        tma_load_3d(sm + kP1 + s * 2 * kBlkBytes + kBlkBytes, &mv, &full1[s], 0, bk * kBlk, unit);
        issued1 = lb + 1;
      }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    for (int r = 0; r < nblk && ok; ++r) {
      const int bk = blk1 - 1 - r, s = r & 1;
      if (lane == 0) {
        if (r >= 2) ok = mbar_wait_or_abort(&empty2[s], ((r >> 1) - 1) & 1, p.timeout_ns, abort_flag);
        if (ok) {
          uint8_t* st = sm + kP2 + s * 4 * kBlkBytes;
          mbar_arrive_expect_tx(&full2[s], 4 * kBlkBytes);
          tma_load_3d(st, &mq, &full2[s], 0, bk * kBlk, unit);
          tma_load_3d(st + kBlkBytes, &mk, &full2[s], 0, bk * kBlk, unit);
          tma_load_3d(st + 2 * kBlkBytes, &mv, &full2[s], 0, bk * kBlk, unit);
          tma_load_3d(st + 3 * kBlkBytes, &mdz, &full2[s], 0, bk * kBlk, unit);
          issued2 = r + 1;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      ok = __all_sync(0xffffffffu, mbar_wait_or_abort(&full2[s], (r >> 1) & 1, p.timeout_ns, abort_flag));
      if (!ok) break;
      seen2 = r + 1;
      // S = tril(Q K^T) and S^T = triu(K Q^T) of each chunk, as packed C fragments.
      const uint32_t sQb = s0 + kP2 + s * 4 * kBlkBytes, sKb = sQb + kBlkBytes;
#pragma unroll 1
      for (int u = 0; u < 4; ++u) {
        const uint32_t sQ = sQb + u * kTileBytes, sK = sKb + u * kTileBytes;
        float sa[2][4] = {}, sb[2][4] = {};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint32_t qa[4], ka[4], rq[4], rk[4];
          ldsm_x4(qa, sQ + swz128(((mi & 1) << 3) + mr, 2 * k + (mi >> 1)));  // Q as A (m = t, k = i)
          ldsm_x4(ka, sK + swz128(((mi & 1) << 3) + mr, 2 * k + (mi >> 1)));  // K as A
          ldsm_x4(rk, sK + swz128(((mi >> 1) << 3) + mr, 2 * k + (mi & 1)));  // K as B (k = i, n = t')
          ldsm_x4(rq, sQ + swz128(((mi >> 1) << 3) + mr, 2 * k + (mi & 1)));  // Q as B
          const uint32_t kb0[2] = {rk[0], rk[1]}, kb1[2] = {rk[2], rk[3]};
          const uint32_t qb0[2] = {rq[0], rq[1]}, qb1[2] = {rq[2], rq[3]};
          mma_bf16_16816(sa[0], qa, kb0);
          mma_bf16_16816(sa[1], qa, kb1);
          mma_bf16_16816(sb[0], ka, qb0);
          mma_bf16_16816(sb[1], ka, qb1);
        }
        // element (row g (+8), column 8nt + 2tg (+1)): keep column <= row in S, column >= row in S^T
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const int c = 8 * nt + 2 * tg;
          if (c > g) sa[nt][0] = 0.f;
          if (c + 1 > g) sa[nt][1] = 0.f;
          if (c > g + 8) sa[nt][2] = 0.f;
          if (c + 1 > g + 8) sa[nt][3] = 0.f;
          if (c < g) sb[nt][0] = 0.f;
          if (c + 1 < g) sb[nt][1] = 0.f;
          if (c < g + 8) sb[nt][2] = 0.f;
          if (c + 1 < g + 8) sb[nt][3] = 0.f;
        }
        uint8_t* dst = sm + kSb + ((s * 4 + u) * 2) * 512 + lane * 16;
        *reinterpret_cast<uint4*>(dst) = make_uint4(pack_bf16(sa[0][0], sa[0][1]), pack_bf16(sa[1][0], sa[1][1]),
                                                    pack_bf16(sa[0][2], sa[0][3]), pack_bf16(sa[1][2], sa[1][3]));
        *reinterpret_cast<uint4*>(dst + 512) = make_uint4(pack_bf16(sb[0][0], sb[0][1]), pack_bf16(sb[1][0], sb[1][1]),
                                                          pack_bf16(sb[0][2], sb[0][3]), pack_bf16(sb[1][2], sb[1][3]));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ready2[s]);
    }
    if (lane == 0) {
      if (!ok) {
        if (!*abort_flag) report_error(p.status, TTT_ERR_TIMEOUT, kWhereBwdProducer, unit);
        *abort_flag = 1;
      }
      // Loads still in flight must land before the CTA may exit.
      for (int bk = (issued1 > 2 ? issued1 - 2 : 0); bk < issued1; ++bk)
        (void)mbar_wait_bounded(&full1[bk & 1], (bk >> 1) & 1, p.timeout_ns);
      for (int r = seen2; r < issued2; ++r) (void)mbar_wait_bounded(&full2[r & 1], (r >> 1) & 1, p.timeout_ns);
    }
    return;
  }

  // ------------------------------------------------------------------ consumers
  const int jw = 16 * warp;
  bool ok = true;
  float Wt[8][4];  // W^T rows j = jw + g (+8), columns i = 8q + 2tg (+1)
  {
    const float* W0 = seg == 0 ? p.W0 + static_cast<size_t>(h) * kD * kD
                               : p.w_starts + (static_cast<size_t>(unit) * (S - 1) + seg - 1) * kD * kD;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int i = 8 * q + 2 * tg;
      Wt[q][0] = __ldcg(W0 + i * kD + jw + g);
      Wt[q][1] = __ldcg(W0 + (i + 1) * kD + jw + g);
      Wt[q][2] = __ldcg(W0 + i * kD + jw + g + 8);
      Wt[q][3] = __ldcg(W0 + (i + 1) * kD + jw + g + 8);
    }
  }
  float* ckpt = p.states + static_cast<size_t>(unit) * nblk_all * kD * kD;  // by absolute block
  auto save_w = [&](float* dst) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int i = 8 * q + 2 * tg;
      dst[i * kD + jw + g] = Wt[q][0];
      dst[(i + 1) * kD + jw + g] = Wt[q][1];
      dst[i * kD + jw + g + 8] = Wt[q][2];
      dst[(i + 1) * kD + jw + g + 8] = Wt[q][3];
    }
  };
  auto load_w = [&](const float* src) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int i = 8 * q + 2 * tg;
      Wt[q][0] = __ldcg(src + i * kD + jw + g);
      Wt[q][1] = __ldcg(src + (i + 1) * kD + jw + g);
      Wt[q][2] = __ldcg(src + i * kD + jw + g + 8);
      Wt[q][3] = __ldcg(src + (i + 1) * kD + jw + g + 8);
    }
  };
  // One chunk of the forward rule on the fragments: E^T = W^T K^T - V^T, W^T -= eta E^T K.
  // Returns E^T (C fragments) and the bf16 A fragments of W^T used.
  auto chunk_forward = [&](uint32_t sK, uint32_t sV, bool update, float (&e)[2][4], uint32_t (&wa)[4][4]) {
    pack_a(Wt, wa);
    float e2[2][4];
    {
      uint32_t vt[4];
      ldsm_x4_t(vt, sV + swz128(((mi >> 1) << 3) + mr, 2 * warp + (mi & 1)));
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        e[nt][0] = -bf16_lo(vt[2 * nt]);
        e[nt][1] = -bf16_hi(vt[2 * nt]);
        e[nt][2] = -bf16_lo(vt[2 * nt + 1]);
        e[nt][3] = -bf16_hi(vt[2 * nt + 1]);
        e2[nt][0] = e2[nt][1] = e2[nt][2] = e2[nt][3] = 0.f;
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t r[4];
      ldsm_x4(r, sK + swz128(((mi >> 1) << 3) + mr, 2 * k + (mi & 1)));
      const uint32_t b0[2] = {r[0], r[1]}, b1[2] = {r[2], r[3]};
      mma_bf16_16816(k < 2 ? e[0] : e2[0], wa[k], b0);
      mma_bf16_16816(k < 2 ? e[1] : e2[1], wa[k], b1);
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) e[nt][r] += e2[nt][r];
    if (update) {
      uint32_t ea[4];
      ea[0] = pack_bf16(-eta * e[0][0], -eta * e[0][1]);
      ea[1] = pack_bf16(-eta * e[0][2], -eta * e[0][3]);
      ea[2] = pack_bf16(-eta * e[1][0], -eta * e[1][1]);
      ea[3] = pack_bf16(-eta * e[1][2], -eta * e[1][3]);
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        uint32_t r[4];
        ldsm_x4_t(r, sK + swz128(((mi & 1) << 3) + mr, 2 * qq + (mi >> 1)));
        const uint32_t b0[2] = {r[0], r[1]}, b1[2] = {r[2], r[3]};
        mma_bf16_16816(Wt[2 * qq], ea, b0);
        mma_bf16_16816(Wt[2 * qq + 1], ea, b1);
      }
    }
  };

  // ---------------------------------------------------------------- pass 1: checkpoints
  for (int lb = 0; lb < nblk; ++lb) {
    const int s = lb & 1, bk = blk0 + lb;
    if (!__all_sync(0xffffffffu, mbar_wait_or_abort(&full1[s], (lb >> 1) & 1, p.timeout_ns, abort_flag))) {
      if (!*abort_flag) report_error(p.status, TTT_ERR_TIMEOUT, kWhereBwdPass1, unit);
      *abort_flag = 1;
      ok = false;
      break;
    }
    save_w(ckpt + static_cast<size_t>(bk) * kD * kD);
    const uint32_t sK = s0 + kP1 + s * 2 * kBlkBytes, sV = sK + kBlkBytes;
    const int nt = min(4, ntiles - 4 * bk);
    for (int u = 0; u < nt; ++u) {
      float e[2][4];
      uint32_t wa[4][4];
      chunk_forward(sK + u * kTileBytes, sV + u * kTileBytes, true, e, wa);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty1[s]);
  }

  // ---------------------------------------------------------------- pass 2: the backward
  float Gt[8][4];  // G^T rows j = jw + g (+8), columns i = 8q + 2tg (+1)
  {
    const float* G0 = seg == S - 1 ? p.dW_out + static_cast<size_t>(unit) * kD * kD
                                   : p.g_ends + (static_cast<size_t>(unit) * (S - 1) + seg) * kD * kD;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int i = 8 * q + 2 * tg;
      Gt[q][0] = __ldcg(G0 + i * kD + jw + g);
      Gt[q][1] = __ldcg(G0 + (i + 1) * kD + jw + g);
      Gt[q][2] = __ldcg(G0 + i * kD + jw + g + 8);
      Gt[q][3] = __ldcg(G0 + (i + 1) * kD + jw + g + 8);
    }
  }
  float deta = 0.f;
  int nsync = 0;  // uses of the consumers' sync barrier (its phase)
  auto sync_all = [&]() -> bool {
    __syncwarp();
    if (lane == 0) mbar_arrive(sync1);
    const bool done = __all_sync(0xffffffffu, mbar_wait_or_abort(sync1, nsync & 1, p.timeout_ns, abort_flag));
    ++nsync;
    return done;
  };
  __nv_bfloat16* dQg = static_cast<__nv_bfloat16*>(p.dQ);
  __nv_bfloat16* dKg = static_cast<__nv_bfloat16*>(p.dK);
  __nv_bfloat16* dVg = static_cast<__nv_bfloat16*>(p.dV);
  const size_t base = static_cast<size_t>(unit) * T * kD;
  int ktile = 0;  // chunks done in pass 2 (which G and dE copy)

  for (int r = 0; ok && r < nblk; ++r) {
    const int bk = blk1 - 1 - r, s = r & 1;
    if (!__all_sync(0xffffffffu, mbar_wait_or_abort(&ready2[s], (r >> 1) & 1, p.timeout_ns, abort_flag))) {
      if (!*abort_flag) report_error(p.status, TTT_ERR_TIMEOUT, kWhereBwdPass2, unit);
      *abort_flag = 1;
      ok = false;
      break;
    }
    const uint32_t sQb = s0 + kP2 + s * 4 * kBlkBytes, sKb = sQb + kBlkBytes, sVb = sQb + 2 * kBlkBytes,
                   sZb = sQb + 3 * kBlkBytes;
    const int nt = min(4, ntiles - 4 * bk);
    // Recompute the block's chunk states and errors from its checkpoint into this block's
    // copies (two sets, by block parity: the other set may still be read for the previous block).
    const uint32_t sWc = s0 + kWc + (r & 1) * kWcBytes, sEc = s0 + kEc + (r & 1) * kEcBytes;
    load_w(ckpt + static_cast<size_t>(bk) * kD * kD);
    for (int u = 0; u < nt; ++u) {
      float e[2][4];
      uint32_t wa[4][4];
      chunk_forward(sKb + u * kTileBytes, sVb + u * kTileBytes, u + 1 < nt, e, wa);
      store_t(sWc + u * kD * kD * 2, wa, warp, lane);  // W_u [i][j], this warp's columns
      const uint32_t ev[4] = {pack_bf16(e[0][0], e[0][1]), pack_bf16(e[0][2], e[0][3]), pack_bf16(e[1][0], e[1][1]),
                              pack_bf16(e[1][2], e[1][3])};
      stsm_x4_t(sEc + u * kTileBytes + swz128(((mi >> 1) << 3) + mr, 2 * warp + (mi & 1)), ev);  // E_u [t][j]
    }
    if (!sync_all()) {  // every warp's columns of W_u and E_u are in place
      ok = false;
      break;
    }

    for (int u = nt - 1; u >= 0; --u, ++ktile) {
      const uint32_t sQ = sQb + u * kTileBytes, sK = sKb + u * kTileBytes, sZ = sZb + u * kTileBytes;
      const uint32_t sW = sWc + u * kD * kD * 2, sE = sEc + u * kTileBytes;
      const uint32_t sG = s0 + kGc + (ktile & 1) * kD * kD * 2, sDE = s0 + kDE + (ktile & 1) * kTileBytes;
      const uint8_t* sfr = sm + kSb + ((s * 4 + u) * 2) * 512 + lane * 16;

      // ---- this warp's output columns j: dE, dV, its part of d eta, and the G update.
      uint32_t ga[4][4];
      pack_a(Gt, ga);
      store_t(sG, ga, warp, lane);  // G [i][j] before this chunk's update, this warp's columns
      float kg[2][4] = {};          // (K G)^T = G^T K^T (rows j, columns t)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t rr[4];
        ldsm_x4(rr, sK + swz128(((mi >> 1) << 3) + mr, 2 * k + (mi & 1)));
        const uint32_t b0[2] = {rr[0], rr[1]}, b1[2] = {rr[2], rr[3]};
        mma_bf16_16816(kg[0], ga[k], b0);
        mma_bf16_16816(kg[1], ga[k], b1);
      }
      uint32_t zt[4];  // dZ^T as A (m = j, k = t')
      ldsm_x4_t(zt, sZ + swz128(((mi >> 1) << 3) + mr, 2 * warp + (mi & 1)));
      float de[2][4];
      {
        const uint4 stv = *reinterpret_cast<const uint4*>(sfr + 512);  // S^T: B[k = t'][n = t] = S[t'][t]
        float zs[2][4] = {};
        const uint32_t b0[2] = {stv.x, stv.y}, b1[2] = {stv.z, stv.w};
        mma_bf16_16816(zs[0], zt, b0);
        mma_bf16_16816(zs[1], zt, b1);
#pragma unroll
        for (int n2 = 0; n2 < 2; ++n2)
#pragma unroll
          for (int q = 0; q < 4; ++q) de[n2][q] = -eta * (kg[n2][q] + zs[n2][q]);
      }
      {  // d eta: -sum(E .* K G) over this warp's columns
        uint32_t et[4];
        ldsm_x4_t(et, sE + swz128(((mi >> 1) << 3) + mr, 2 * warp + (mi & 1)));
#pragma unroll
        for (int n2 = 0; n2 < 2; ++n2)
          deta -= bf16_lo(et[2 * n2]) * kg[n2][0] + bf16_hi(et[2 * n2]) * kg[n2][1] +
                  bf16_lo(et[2 * n2 + 1]) * kg[n2][2] + bf16_hi(et[2 * n2 + 1]) * kg[n2][3];
      }
      const uint32_t dea[4] = {pack_bf16(de[0][0], de[0][1]), pack_bf16(de[0][2], de[0][3]),
                               pack_bf16(de[1][0], de[1][1]), pack_bf16(de[1][2], de[1][3])};
      stsm_x4_t(sDE + swz128(((mi >> 1) << 3) + mr, 2 * warp + (mi & 1)), dea);  // dE [t][j]
      // G^T += dZ^T Q + dE^T K (the copy in sG keeps the G this chunk's products need).
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        uint32_t rq[4], rk[4];
        ldsm_x4_t(rq, sQ + swz128(((mi & 1) << 3) + mr, 2 * qq + (mi >> 1)));
        ldsm_x4_t(rk, sK + swz128(((mi & 1) << 3) + mr, 2 * qq + (mi >> 1)));
        const uint32_t q0[2] = {rq[0], rq[1]}, q1[2] = {rq[2], rq[3]};
        const uint32_t k0[2] = {rk[0], rk[1]}, k1[2] = {rk[2], rk[3]};
        mma_bf16_16816(Gt[2 * qq], zt, q0);
        mma_bf16_16816(Gt[2 * qq + 1], zt, q1);
        mma_bf16_16816(Gt[2 * qq], dea, k0);
        mma_bf16_16816(Gt[2 * qq + 1], dea, k1);
      }
      const int tok0 = 64 * bk + 16 * u;
      {  // dV = -dE for this warp's columns
        __syncwarp();
        const int tok = tok0 + (lane >> 1);
        uint4 x = *reinterpret_cast<const uint4*>(sm + (sDE - s0) + swz128(lane >> 1, 2 * warp + (lane & 1)));
        x.x ^= 0x80008000u;
        x.y ^= 0x80008000u;
        x.z ^= 0x80008000u;
        x.w ^= 0x80008000u;
        if (tok < T) *reinterpret_cast<uint4*>(dVg + base + static_cast<size_t>(tok) * kD + jw + 8 * (lane & 1)) = x;
      }
      if (!sync_all()) {  // every warp's columns of G and dE are in place
        ok = false;
        break;
      }

      // ---- this warp's band of input features i in [16w, 16w + 16): P, dQ, dK over all columns.
      uint32_t za[4][4];  // dZ as A (m = t, k = j), k-step k: j in [16k, 16k + 16)
#pragma unroll
      for (int k = 0; k < 4; ++k) ldsm_x4(za[k], sZ + swz128(((mi & 1) << 3) + mr, 2 * k + (mi >> 1)));
      uint32_t pa[4], pta[4];
      {  // P = -eta tril(dZ E^T), the full 16 x 16 (every warp forms it)
        float pc[2][4] = {};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint32_t rr[4];
          ldsm_x4(rr, sE + swz128(((mi >> 1) << 3) + mr, 2 * k + (mi & 1)));  // E as B (k = j, n = t')
          const uint32_t b0[2] = {rr[0], rr[1]}, b1[2] = {rr[2], rr[3]};
          mma_bf16_16816(pc[0], za[k], b0);
          mma_bf16_16816(pc[1], za[k], b1);
        }
        if (warp == 0) {  // d eta: -sum(S .* dZ E^T), once
          float sf[2][4];
          unpack4(*reinterpret_cast<const uint4*>(sfr), sf);
#pragma unroll
          for (int n2 = 0; n2 < 2; ++n2)
#pragma unroll
            for (int q = 0; q < 4; ++q) deta -= sf[n2][q] * pc[n2][q];
        }
#pragma unroll
        for (int n2 = 0; n2 < 2; ++n2) {  // keep t' <= t, scale by -eta
          const int c = 8 * n2 + 2 * tg;
          pc[n2][0] = c > g ? 0.f : -eta * pc[n2][0];
          pc[n2][1] = c + 1 > g ? 0.f : -eta * pc[n2][1];
          pc[n2][2] = c > g + 8 ? 0.f : -eta * pc[n2][2];
          pc[n2][3] = c + 1 > g + 8 ? 0.f : -eta * pc[n2][3];
        }
        pa[0] = pack_bf16(pc[0][0], pc[0][1]);
        pa[1] = pack_bf16(pc[0][2], pc[0][3]);
        pa[2] = pack_bf16(pc[1][0], pc[1][1]);
        pa[3] = pack_bf16(pc[1][2], pc[1][3]);
        pta[0] = movm_t(pa[0]);  // P^T's 8 x 8 blocks are the transposed blocks of P
        pta[1] = movm_t(pa[2]);
        pta[2] = movm_t(pa[1]);
        pta[3] = movm_t(pa[3]);
      }
      float oq[2][4] = {}, ok2[2][4] = {};
      {
        uint32_t rk[4], rq[4];  // K and Q as B (k = t', n = i in the band)
        ldsm_x4_t(rk, sK + swz128(((mi & 1) << 3) + mr, 2 * warp + (mi >> 1)));
        ldsm_x4_t(rq, sQ + swz128(((mi & 1) << 3) + mr, 2 * warp + (mi >> 1)));
        const uint32_t k0[2] = {rk[0], rk[1]}, k1[2] = {rk[2], rk[3]};
        const uint32_t q0[2] = {rq[0], rq[1]}, q1[2] = {rq[2], rq[3]};
        mma_bf16_16816(oq[0], pa, k0);   // P K
        mma_bf16_16816(oq[1], pa, k1);
        mma_bf16_16816(ok2[0], pta, q0); // P^T Q
        mma_bf16_16816(ok2[1], pta, q1);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {  // sums over the columns j in [16k, 16k + 16)
        uint32_t rw[4], rg[4], ea[4], da[4];
        ldsm_x4(rw, sW + swz128(jw + ((mi >> 1) << 3) + mr, 2 * k + (mi & 1)));  // W rows i as B (k = j, n = i)
        ldsm_x4(rg, sG + swz128(jw + ((mi >> 1) << 3) + mr, 2 * k + (mi & 1)));  // G rows i as B
        ldsm_x4(ea, sE + swz128(((mi & 1) << 3) + mr, 2 * k + (mi >> 1)));       // E as A (m = t, k = j)
        ldsm_x4(da, sDE + swz128(((mi & 1) << 3) + mr, 2 * k + (mi >> 1)));      // dE as A
#pragma unroll
        for (int q = 0; q < 4; ++q) ea[q] = pack_bf16(-eta * bf16_lo(ea[q]), -eta * bf16_hi(ea[q]));
        const uint32_t w0[2] = {rw[0], rw[1]}, w1[2] = {rw[2], rw[3]};
        const uint32_t g0[2] = {rg[0], rg[1]}, g1[2] = {rg[2], rg[3]};
        mma_bf16_16816(oq[0], za[k], w0);  // dZ W^T
        mma_bf16_16816(oq[1], za[k], w1);
        mma_bf16_16816(ok2[0], da, w0);    // dE W^T
        mma_bf16_16816(ok2[1], da, w1);
        mma_bf16_16816(ok2[0], ea, g0);    // -eta E G^T
        mma_bf16_16816(ok2[1], ea, g1);
      }
      // Out through the warp's staging tile ([t][16 i], 32-byte rows), one 16-byte store per lane.
      auto emit = [&](const float (&o)[2][4], __nv_bfloat16* dst, int buf) {
        uint8_t* stg = sm + kOut + (warp * 2 + buf) * 512;
        const uint32_t v[4] = {pack_bf16(o[0][0], o[0][1]), pack_bf16(o[0][2], o[0][3]), pack_bf16(o[1][0], o[1][1]),
                               pack_bf16(o[1][2], o[1][3])};
        stsm_x4(smem_u32(stg) + ((mi & 1) * 8 + mr) * 32 + (mi >> 1) * 16, v);
        __syncwarp();
        const int tok = tok0 + (lane >> 1);
        const uint4 x = *reinterpret_cast<const uint4*>(stg + (lane >> 1) * 32 + (lane & 1) * 16);
        if (tok < T) *reinterpret_cast<uint4*>(dst + base + static_cast<size_t>(tok) * kD + jw + 8 * (lane & 1)) = x;
      };
      emit(oq, dQg, 0);
      emit(ok2, dKg, 1);
      __syncwarp();
    }
    if (!ok) break;
    // Every read of this block's tiles is done: hand the stage back.
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty2[s]);
  }
  if (!ok && !*abort_flag) report_error(p.status, TTT_ERR_TIMEOUT, kWhereBwdSync, unit);
  if (!ok) *abort_flag = 1;

  // dW0 share of this unit (G after the first chunk: the first segment's CTA only) and d eta.
  float* part = p.partial + (static_cast<size_t>(unit) * S + seg) * (kD * kD + 1);
  const float keep = seg == 0 ? 1.f : 0.f;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int i = 8 * q + 2 * tg;
    part[i * kD + jw + g] = keep * Gt[q][0];
    part[(i + 1) * kD + jw + g] = keep * Gt[q][1];
    part[i * kD + jw + g + 8] = keep * Gt[q][2];
    part[(i + 1) * kD + jw + g + 8] = keep * Gt[q][3];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) deta += __shfl_xor_sync(0xffffffffu, deta, o);
  float* red = reinterpret_cast<float*>(sm + kRed);
  if (lane == 0) red[warp] = deta;
  asm volatile("bar.sync 1, %0;" ::"n"(kWarps * 32) : "memory");  // the four consumer warps only
  if (threadIdx.x == 0) part[kD * kD] = red[0] + red[1] + red[2] + red[3];
}

}  // namespace

bool linear_bwd_mma_supported(int d, int b, bool bf16) { return bf16 && d == kD && b == kTile; }

int linear_bwd_mma_rows() { return kBlk; }

cudaError_t launch_linear_bwd_mma(const LinearBwdParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                                  const CUtensorMap& mv, const CUtensorMap& mdz, cudaStream_t stream) {
  if (p.units == 0) return cudaSuccess;
  auto kern = p.bseg_count > 1 ? linear_bwd_mma_kernel<true> : linear_bwd_mma_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<p.units * p.bseg_count, kThreads, kSmemBytes, stream>>>(mq, mk, mv, mdz, p);
  return cudaGetLastError();
}

}  // namespace ttt
