// TTT-Linear forward, bf16 inputs, d = 64, chunk b a multiple of 16:
// one CTA per (batch row, head), W resident in registers across the sequence.
//
// Method ("5 · TestingTime 训练与长上下文", sections 1.1 and 2.3; "Test-Time
// Training (TTT) guide", section 3): for chunk c with start state Wa,
//   E = K_c Wa - V_c,   Z_c = Q_c Wa - eta tril(Q_c K_c^T) E,   W = Wa - eta K_c^T E.
//
// Design. The loss 1/2||k W - v||^2 splits over the output columns j of W, so
// column j of W evolves on its own: W[:, j] -= eta K^T (K W[:, j] - V[:, j]).
// Each of the 4 consumer warps owns 16 output columns and keeps its slice of
// W^T (16 x 64 fp32) as mma.sync accumulator fragments. Everything is written
// transposed so that no fragment ever needs a transpose:
//   E^T  = W^T K^T - V^T          (M = 16 columns j, N = 16 tokens, K = 64)
//   W^T += (-eta E^T) K           (M = 16, N = 64, K = 16 tokens)
//   Z^T  = W^T Q^T + (-eta E^T) S^T,   S = tril(Q K^T)
// The accumulator (C) fragment of an m16n8 product has exactly the register
// layout of the A operand of the next m16n8k16 product, so W^T -> A(W^T),
// E^T -> A(E^T) and S -> B(S^T) stay in registers. The per-chunk serial chain
// is two dependent MMA rounds and a few conversions.
//
// A chunk larger than 16 tokens is walked in 16-token tiles: E of every tile
// uses the chunk-start snapshot of W (its bf16 fragments are kept), while the
// read-out of tile u uses the running W, which already holds the gradients of
// the chunk's earlier tiles; that equals Q Wa - eta tril(Q K^T) E restricted
// to the tile, because Q_u Wa - eta sum_{u'<u} (Q_u K_u'^T) E_u' = Q_u W_run.
//
// Data movement: a producer warp streams the Q, K, V tiles (16 x 64 bf16,
// 2 KB each) with TMA into a 6-stage ring (128-byte swizzle, so ldmatrix is
// conflict-free) and forms each tile's S = tril(Q K^T) once for the four
// consumer warps; Z leaves through a transposing stmatrix into a small staging
// tile per warp and one 16-byte store per lane. Every wait is bounded in
// wall-clock time.
//
// Segments: with p.seg_count > 1 a CTA serves one segment of one unit, starting
// from the state the combine step of linear_seg.cu computed for it (W0 for the
// first segment); only the last segment writes the final state.
#include "ttt_device.cuh"
#include "kernels.h"

namespace ttt {
namespace {

constexpr int kD = 64;
constexpr int kTile = 16;
constexpr int kStages = 6;
constexpr int kWarps = 4;                     // consumer warps; one more produces
constexpr int kThreads = (kWarps + 1) * 32;
constexpr int kTileBytes = kTile * kD * 2;    // 2048
constexpr int kStageBytes = 3 * kTileBytes;   // Q, K, V
constexpr int kZOff = kStages * kStageBytes;  // 24576
constexpr int kZBytes = kTile * 16 * 2;       // 512 per warp and buffer
constexpr int kSOff = kZOff + kWarps * 2 * kZBytes;  // per stage: S^T B fragments, 16 bytes per lane
constexpr int kSBytes = 32 * 16;
constexpr int kBarOff = kSOff + kStages * kSBytes;
constexpr int kAbortOff = kBarOff + 3 * kStages * 8;
constexpr int kSmemBytes = kAbortOff + 16 + 1024;  // + slack to align the base to 1024
static_assert(kSmemBytes <= 48 * 1024, "no opt-in to more dynamic shared memory");
static_assert(3 * kSmemBytes <= 227 * 1024, "three CTAs per SM");

enum : int { kWhereProducer = 1, kWhereConsumer = 2 };

// kTileChunk: every 16-token tile is a whole chunk (b = 16), so the chunk-start
// copy of W^T is the running one and no second copy is kept.
template <bool kTileChunk>
__global__ void __launch_bounds__(kThreads, 3)
    linear_mma_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                      const __grid_constant__ CUtensorMap mv,
                      LinearParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* empty = full + kStages;
  uint64_t* sready = empty + kStages;  // the tile's S fragments are written
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortOff);

  const int unit = blockIdx.x / p.seg_num;
  const int seg = p.seg_first + blockIdx.x % p.seg_num;
  const int h = unit % p.H;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int t0 = seg * p.seg_len;  // a multiple of b: segments start on a chunk boundary
  const int t1 = min(p.T, t0 + p.seg_len);
  const int num_tiles = (t1 - t0 + kTile - 1) / kTile;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps);
      mbar_init(&sready[s], 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kWarps) {
    // ------------------------------------------------------------ producer
    // Lane 0 streams the tiles; the whole warp forms each tile's S = tril(Q K^T)
    // once for the four consumer warps, as the B fragments of S^T they use.
    const int g = lane >> 2, tg = lane & 3, mi = lane >> 3, mr = lane & 7;
    int issued = 0;  // lane 0
    auto load = [&](int u) {
      const int s = u % kStages;
      mbar_arrive_expect_tx(&full[s], kStageBytes);
      uint8_t* st = smem + s * kStageBytes;
      tma_load_3d(st, &mq, &full[s], 0, t0 + u * kTile, unit);
      tma_load_3d(st + kTileBytes, &mk, &full[s], 0, t0 + u * kTile, unit);
      tma_load_3d(st + 2 * kTileBytes, &mv, &full[s], 0, t0 + u * kTile, unit);
      ++issued;
    };
    if (lane == 0) {
      prefetch_tmap(&mq);
      prefetch_tmap(&mk);
      prefetch_tmap(&mv);
      if (!p.inject_stall)
        for (int u = 0; u < min(kStages, num_tiles); ++u) load(u);
    }
    bool ok = true;
    for (int u = 0; u < num_tiles; ++u) {
      const int s = u % kStages;
      if (!mbar_wait_or_abort(&full[s], (u / kStages) & 1, p.timeout_ns, abort_flag)) {
        ok = false;
        break;
      }
      const uint32_t sQ = smem_u32(smem + s * kStageBytes);
      const uint32_t sK = sQ + kTileBytes;
      float sacc[2][4] = {};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t qa[4], r[4];
        ldsm_x4(qa, sQ + swz128(((mi & 1) << 3) + mr, 2 * k + (mi >> 1)));  // Q: A (m = t, k = i)
        ldsm_x4(r, sK + swz128(((mi >> 1) << 3) + mr, 2 * k + (mi & 1)));   // K: B (k = i, n = t')
        const uint32_t b0[2] = {r[0], r[1]}, b1[2] = {r[2], r[3]};
        mma_bf16_16816(sacc[0], qa, b0);
        mma_bf16_16816(sacc[1], qa, b1);
      }
      // Element (t, t') with t = g (+8), t' = 8nt + 2tg (+1); keep t' <= t (each token
      // sees its own gradient).
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int c = 8 * nt + 2 * tg;
        if (c > g) sacc[nt][0] = 0.f;
        if (c + 1 > g) sacc[nt][1] = 0.f;
        if (c > g + 8) sacc[nt][2] = 0.f;
        if (c + 1 > g + 8) sacc[nt][3] = 0.f;
      }
      // S's C fragment (rows t, columns t') is the B fragment (k = t', n = t) of S^T.
      *reinterpret_cast<uint4*>(smem + kSOff + s * kSBytes + lane * 16) =
          make_uint4(pack_bf16(sacc[0][0], sacc[0][1]), pack_bf16(sacc[1][0], sacc[1][1]),
                     pack_bf16(sacc[0][2], sacc[0][3]), pack_bf16(sacc[1][2], sacc[1][3]));
      __syncwarp();
      if (lane == 0) mbar_arrive(&sready[s]);
      // Refill the stage of tile u - 1 once the consumers have released it.
      const int v = u - 1 + kStages;
      if (u >= 1 && v < num_tiles && !p.inject_stall) {
        if (lane == 0) {
          ok = mbar_wait_or_abort(&empty[(u - 1) % kStages], ((u - 1) / kStages) & 1, p.timeout_ns, abort_flag);
          if (ok) load(v);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
    }
    if (lane == 0) {
      if (!ok) {
        if (!*abort_flag) report_error(p.status, TTT_ERR_TIMEOUT, kWhereProducer, unit);
        *abort_flag = 1;
      }
      // Loads still in flight must land before the CTA may exit.
      for (int u = (issued > kStages ? issued - kStages : 0); u < issued; ++u)
        (void)mbar_wait_bounded(&full[u % kStages], (u / kStages) & 1, p.timeout_ns);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2;   // fragment row group
  const int tg = lane & 3;   // thread in group
  const int jw = 16 * warp;  // first output column of this warp
  const int mi = lane >> 3;  // ldmatrix/stmatrix: which 8x8 matrix this lane addresses
  const int mr = lane & 7;   // ... and which of its rows
  const float neta = -p.eta[h];
  __nv_bfloat16* Zg = static_cast<__nv_bfloat16*>(p.Z);

  // W^T fragments: Wt[q] covers input columns i in [8q, 8q+8) of rows j = jw+g, jw+g+8.
  float Wt[8][4];
  {
    const float* W0 = seg == 0 ? p.W0 + static_cast<size_t>(h) * kD * kD
                               : p.seg_starts + (static_cast<size_t>(unit) * (p.seg_count - 1) + seg - 1) * kD * kD;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int i = 8 * q + 2 * tg;
      Wt[q][0] = W0[i * kD + jw + g];
      Wt[q][1] = W0[(i + 1) * kD + jw + g];
      Wt[q][2] = W0[i * kD + jw + g + 8];
      Wt[q][3] = W0[(i + 1) * kD + jw + g + 8];
    }
  }

  uint32_t wr[4][4];  // bf16 A fragments of the running W^T at the tile start (k-step s: i in [16s, 16s+16))
  uint32_t wa[4][4];  // ... and of the chunk-start W^T (not kept when every tile is a chunk)

  for (int u = 0; u < num_tiles; ++u) {
    const int s = u % kStages;
    // The producer raises sready only after it has seen the tile land (full) and
    // read it, so sready alone orders this warp's reads after the TMA writes.
    if (!mbar_wait_or_abort(&sready[s], (u / kStages) & 1, p.timeout_ns, abort_flag)) {
      if (!*abort_flag) report_error(p.status, TTT_ERR_TIMEOUT, kWhereConsumer, unit);
      *abort_flag = 1;
      break;
    }
    // S^T's B fragments for this lane, formed by the producer warp.
    const uint4 sv = *reinterpret_cast<const uint4*>(smem + kSOff + s * kSBytes + lane * 16);
    const uint32_t sQ = smem_u32(smem + s * kStageBytes);
    const uint32_t sK = sQ + kTileBytes;
    const uint32_t sV = sQ + 2 * kTileBytes;

#pragma unroll
    for (int k = 0; k < 4; ++k) {
      wr[k][0] = pack_bf16(Wt[2 * k][0], Wt[2 * k][1]);
      wr[k][1] = pack_bf16(Wt[2 * k][2], Wt[2 * k][3]);
      wr[k][2] = pack_bf16(Wt[2 * k + 1][0], Wt[2 * k + 1][1]);
      wr[k][3] = pack_bf16(Wt[2 * k + 1][2], Wt[2 * k + 1][3]);
    }
    if constexpr (!kTileChunk) {
      if (((u * kTile) % p.b) == 0) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int r = 0; r < 4; ++r) wa[k][r] = wr[k][r];
      }
    }

    // -V^T as the accumulator of E^T. ldmatrix.trans of the V tile's 8x8 blocks
    // (rows t, columns j) hands lane (g, tg) the pair V[2tg..2tg+1][j = g], which
    // is the C-fragment pair (row j, columns t) of E^T.
    float e[2][4], e2[2][4];
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

    // K as the B operand (k = i, n = t): kb[nt][k] for tokens [8nt, 8nt+8), i in [16k, 16k+16).
    uint32_t kb[2][4][2];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t r[4];
      ldsm_x4(r, sK + swz128(((mi >> 1) << 3) + mr, 2 * k + (mi & 1)));
      kb[0][k][0] = r[0];
      kb[0][k][1] = r[1];
      kb[1][k][0] = r[2];
      kb[1][k][1] = r[3];
    }
    // E^T = W_a^T K^T - V^T, in two independent partial sums to shorten the chain.
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) mma_bf16_16816(k < 2 ? e[nt] : e2[nt], kTileChunk ? wr[k] : wa[k], kb[nt][k]);

    // K^T-side B operand for the update (k = t, n = i): kbt[q] for i in [8q, 8q+8).
    uint32_t kbt[8][2];
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) {
      uint32_t r[4];
      ldsm_x4_t(r, sK + swz128(((mi & 1) << 3) + mr, 2 * qq + (mi >> 1)));
      kbt[2 * qq][0] = r[0];
      kbt[2 * qq][1] = r[1];
      kbt[2 * qq + 1][0] = r[2];
      kbt[2 * qq + 1][1] = r[3];
    }

#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      e[nt][0] += e2[nt][0];
      e[nt][1] += e2[nt][1];
      e[nt][2] += e2[nt][2];
      e[nt][3] += e2[nt][3];
    }
    // -eta E^T as the A operand (m = j, k = t).
    uint32_t ea[4];
    ea[0] = pack_bf16(neta * e[0][0], neta * e[0][1]);
    ea[1] = pack_bf16(neta * e[0][2], neta * e[0][3]);
    ea[2] = pack_bf16(neta * e[1][0], neta * e[1][1]);
    ea[3] = pack_bf16(neta * e[1][2], neta * e[1][3]);

    // W^T += (-eta E^T) K: the state update of the chunk's gradient step.
#pragma unroll
    for (int q = 0; q < 8; ++q) mma_bf16_16816(Wt[q], ea, kbt[q]);

    // The read-out's products come after the update, so that the update (the serial
    // chain to the next tile) is issued first; they use the tile-start copy wr.
    // Read-out part 1: Z^T = W_run^T Q^T (Q as B operand, like K).
    float z[2][4] = {};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t r[4];
      ldsm_x4(r, sQ + swz128(((mi >> 1) << 3) + mr, 2 * k + (mi & 1)));
      uint32_t qb0[2] = {r[0], r[1]}, qb1[2] = {r[2], r[3]};
      mma_bf16_16816(z[0], wr[k], qb0);
      mma_bf16_16816(z[1], wr[k], qb1);
    }

    const uint32_t sb0[2] = {sv.x, sv.y}, sb1[2] = {sv.z, sv.w};
    // Read-out part 2: Z^T += (-eta E^T) S^T.
    mma_bf16_16816(z[0], ea, sb0);
    mma_bf16_16816(z[1], ea, sb1);

    // Hand the stage back to the producer, whose next TMA load overwrites it. Only
    // now has every register loaded from it (K^T for the update, S^T) been consumed,
    // so no load from the stage is still outstanding; the proxy fence orders these
    // generic-proxy reads before that async-proxy write. (Releasing it right after
    // issuing the last ldmatrix let a delayed load read the next tile's K.)
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);

    // Z^T (rows j, columns t) -> Z[t][j] (16 x 16 bf16) in the warp's staging tile
    // by a transposing stmatrix, then one 16-byte store per lane: rows of 32 bytes.
    uint8_t* zbuf = smem + kZOff + (warp * 2 + (u & 1)) * kZBytes;
    {
      uint32_t zr[4] = {pack_bf16(z[0][0], z[0][1]), pack_bf16(z[0][2], z[0][3]),
                        pack_bf16(z[1][0], z[1][1]), pack_bf16(z[1][2], z[1][3])};
      stsm_x4_t(smem_u32(zbuf) + (((mi >> 1) << 3) + mr) * 32 + (mi & 1) * 16, zr);
    }
    __syncwarp();
    {
      const int tok = t0 + u * kTile + (lane >> 1);
      const uint4 zv = *reinterpret_cast<const uint4*>(zbuf + (lane >> 1) * 32 + (lane & 1) * 16);
      if (tok < t1)
        *reinterpret_cast<uint4*>(Zg + (static_cast<size_t>(unit) * p.T + tok) * kD + jw + 8 * (lane & 1)) = zv;
    }
  }
  if (seg != p.seg_count - 1) return;

  // Final state, W_out[unit][i][j].
  float* Wo = p.W_out + static_cast<size_t>(unit) * kD * kD;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int i = 8 * q + 2 * tg;
    Wo[i * kD + jw + g] = Wt[q][0];
    Wo[(i + 1) * kD + jw + g] = Wt[q][1];
    Wo[i * kD + jw + g + 8] = Wt[q][2];
    Wo[(i + 1) * kD + jw + g + 8] = Wt[q][3];
  }
}

}  // namespace

bool linear_mma_supported(const LinearParams& p) { return p.d == kD && p.b % kTile == 0 && p.bf16; }

cudaError_t launch_linear_mma(const LinearParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                              const CUtensorMap& mv, cudaStream_t stream) {
  if (p.units == 0) return cudaSuccess;
  if (p.seg_num == 0) return cudaSuccess;
  if (p.b == kTile)
    linear_mma_kernel<true><<<p.units * p.seg_num, kThreads, kSmemBytes, stream>>>(mq, mk, mv, p);
  else
    linear_mma_kernel<false><<<p.units * p.seg_num, kThreads, kSmemBytes, stream>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

int linear_mma_tile_rows() { return kTile; }

}  // namespace ttt
