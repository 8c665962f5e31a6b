// Segment-parallel backward of the chunked TTT-Linear scan (bf16, d = 64,
// b = 16): the pieces that let linear_bwd_mma.cu run one CTA per (unit,
// segment) instead of one per unit.
//
// Each chunk's read-out is affine in its start state ("5 · TestingTime 训练与长
// 上下文", sections 1.1 and 4; the pages do not write it this way, it is exact
// algebra on the chunk rule): with A_c = I - eta K_c^T K_c,
//   W_{c+1} = A_c W_c + eta K_c^T V_c,   Z_c = P_c W_c + (terms free of W),
//   P_c = Q_c - eta S_c K_c,  S_c = tril(Q_c K_c^T).
// So the gradient of a segment's start state is
//   G_start(s) = A_s^T G_end(s) + H_s,   H_s = sum_c Phi_c^T P_c^T dZ_c,
// where Phi_c = A_{c-1} ... A_{c0} carries the segment's start state to chunk c
// and A_s is Phi at the segment's end. Both depend on Q, K, dZ only, not on W:
//   linear_bwd_hmap_kernel runs the forward chunk rule from Phi = I with V = 0.
//   Then E_c = K_c Phi_c, Phi_{c+1} = Phi_c - eta K_c^T E_c = A_c Phi_c, and the
//   dual-form read-out Zhat_c = Q_c Phi_c - eta S_c E_c is exactly P_c Phi_c,
//   so H_s = sum over tokens of Zhat^T dZ: one more rank-16 product per tile on
//   the accumulator fragments of the read-out kernel's layout (linear_mma.cu).
//   It writes H_s and A_s for segments 1..S-1, all at once.
//   linear_bwd_rcombine_kernel: G_end(S-1) = dW_out and, last segment first,
//   G_end(s - 1) = A_s^T G_end(s) + H_s in fp32 (per unit and group of 8
//   columns: the product is column-separable).
// With the forward's start states W_start(s) (the segment affine maps and their
// combine, linear_seg_wy.cu / linear_seg.cu), every segment then runs the
// backward on its own range.
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
constexpr int kStageBytes = 3 * kTileBytes;   // Q, K, dZ
constexpr int kSOff = kStages * kStageBytes;  // per stage: S^T B fragments, 16 bytes per lane
constexpr int kSBytes = 32 * 16;
constexpr int kBarOff = kSOff + kStages * kSBytes;
constexpr int kAbortOff = kBarOff + 3 * kStages * 8;
constexpr int kSmemBytes = kAbortOff + 16 + 1024;  // + slack to align the base to 1024
static_assert(kSmemBytes <= 48 * 1024, "no opt-in to more dynamic shared memory");

enum : int { kWhereHmapProducer = 30, kWhereHmapConsumer = 31 };

__global__ void __launch_bounds__(kThreads, 2)
    linear_bwd_hmap_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                           const __grid_constant__ CUtensorMap mdz, LinearBwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* empty = full + kStages;
  uint64_t* sready = empty + kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortOff);

  const int nseg = p.bseg_count - 1;             // segments 1 .. S-1
  const int unit = blockIdx.x / nseg;
  const int seg = 1 + blockIdx.x % nseg;
  const int h = unit % p.H;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int t0 = seg * p.bseg_len;
  const int t1 = min(p.T, t0 + p.bseg_len);
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
    // ------------------------------------------------------------ producer: TMA ring and S
    const int g = lane >> 2, tg = lane & 3, mi = lane >> 3, mr = lane & 7;
    int issued = 0;
    auto load = [&](int u) {
      const int s = u % kStages;
      mbar_arrive_expect_tx(&full[s], kStageBytes);
      uint8_t* st = smem + s * kStageBytes;
      tma_load_3d(st, &mq, &full[s], 0, t0 + u * kTile, unit);
      tma_load_3d(st + kTileBytes, &mk, &full[s], 0, t0 + u * kTile, unit);
      tma_load_3d(st + 2 * kTileBytes, &mdz, &full[s], 0, t0 + u * kTile, unit);
      ++issued;
    };
    if (lane == 0) {
      prefetch_tmap(&mq);
      prefetch_tmap(&mk);
      prefetch_tmap(&mdz);
      for (int u = 0; u < min(kStages, num_tiles); ++u) load(u);
    }
    bool ok = true;
    for (int u = 0; u < num_tiles; ++u) {
      const int s = u % kStages;
      if (!__all_sync(0xffffffffu, mbar_wait_or_abort(&full[s], (u / kStages) & 1, p.timeout_ns, abort_flag))) {
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
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {  // keep t' <= t
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
      const int v = u - 1 + kStages;  // refill the stage of tile u - 1 once it is released
      if (u >= 1 && v < num_tiles) {
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
        if (!*abort_flag) report_error(p.status, TTT_ERR_TIMEOUT, kWhereHmapProducer, unit);
        *abort_flag = 1;
      }
      for (int u = (issued > kStages ? issued - kStages : 0); u < issued; ++u)
        (void)mbar_wait_bounded(&full[u % kStages], (u / kStages) & 1, p.timeout_ns);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2;   // fragment row group
  const int tg = lane & 3;   // thread in group
  const int jw = 16 * warp;  // this warp's 16 columns of Phi (and rows of H)
  const int mi = lane >> 3;
  const int mr = lane & 7;
  const float neta = -p.eta[h];

  // Phi^T fragments, from the identity: Pt[q] covers input columns i in [8q, 8q+8) of rows j = jw+g, +8.
  float Pt[8][4];
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int i = 8 * q + 2 * tg;
    Pt[q][0] = i == jw + g ? 1.f : 0.f;
    Pt[q][1] = i + 1 == jw + g ? 1.f : 0.f;
    Pt[q][2] = i == jw + g + 8 ? 1.f : 0.f;
    Pt[q][3] = i + 1 == jw + g + 8 ? 1.f : 0.f;
  }
  // H's rows j = jw + g (+8), columns n = 8q + 2tg (+1): sum over tokens of Zhat[t][j] dZ[t][n].
  float Hc[8][4] = {};

  bool ok = true;
  for (int u = 0; u < num_tiles; ++u) {
    const int s = u % kStages;
    if (!__all_sync(0xffffffffu, mbar_wait_or_abort(&sready[s], (u / kStages) & 1, p.timeout_ns, abort_flag))) {
      ok = false;
      break;
    }
    const uint4 sv = *reinterpret_cast<const uint4*>(smem + kSOff + s * kSBytes + lane * 16);
    const uint32_t sQ = smem_u32(smem + s * kStageBytes);
    const uint32_t sK = sQ + kTileBytes;
    const uint32_t sDZ = sQ + 2 * kTileBytes;

    uint32_t wr[4][4];  // bf16 A fragments of Phi^T at the tile start
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      wr[k][0] = pack_bf16(Pt[2 * k][0], Pt[2 * k][1]);
      wr[k][1] = pack_bf16(Pt[2 * k][2], Pt[2 * k][3]);
      wr[k][2] = pack_bf16(Pt[2 * k + 1][0], Pt[2 * k + 1][1]);
      wr[k][3] = pack_bf16(Pt[2 * k + 1][2], Pt[2 * k + 1][3]);
    }
    // E^T = Phi^T K^T (no values: V = 0), in two partial sums.
    float e[2][4] = {}, e2[2][4] = {};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t r[4];
      ldsm_x4(r, sK + swz128(((mi >> 1) << 3) + mr, 2 * k + (mi & 1)));
      const uint32_t b0[2] = {r[0], r[1]}, b1[2] = {r[2], r[3]};
      mma_bf16_16816(k < 2 ? e[0] : e2[0], wr[k], b0);
      mma_bf16_16816(k < 2 ? e[1] : e2[1], wr[k], b1);
    }
    uint32_t kbt[8][2];  // K as the B operand (k = t, n = i) of the update
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
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) e[nt][r] += e2[nt][r];
    uint32_t ea[4];  // -eta E^T as the A operand (m = j, k = t)
    ea[0] = pack_bf16(neta * e[0][0], neta * e[0][1]);
    ea[1] = pack_bf16(neta * e[0][2], neta * e[0][3]);
    ea[2] = pack_bf16(neta * e[1][0], neta * e[1][1]);
    ea[3] = pack_bf16(neta * e[1][2], neta * e[1][3]);
    // Phi^T += (-eta E^T) K: the chunk's update of the propagator.
#pragma unroll
    for (int q = 0; q < 8; ++q) mma_bf16_16816(Pt[q], ea, kbt[q]);

    // Zhat^T = Phi^T Q^T - eta E^T S^T, with the tile-start copy wr.
    float z[2][4] = {};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t r[4];
      ldsm_x4(r, sQ + swz128(((mi >> 1) << 3) + mr, 2 * k + (mi & 1)));
      const uint32_t qb0[2] = {r[0], r[1]}, qb1[2] = {r[2], r[3]};
      mma_bf16_16816(z[0], wr[k], qb0);
      mma_bf16_16816(z[1], wr[k], qb1);
    }
    const uint32_t sb0[2] = {sv.x, sv.y}, sb1[2] = {sv.z, sv.w};
    mma_bf16_16816(z[0], ea, sb0);
    mma_bf16_16816(z[1], ea, sb1);

    // H += Zhat^T dZ: Zhat^T's C fragment (rows j, columns t) is the A operand (m = j, k = t);
    // dZ as the B operand (k = t, n = feature) by the transposing loads used for K above.
    const uint32_t za[4] = {pack_bf16(z[0][0], z[0][1]), pack_bf16(z[0][2], z[0][3]), pack_bf16(z[1][0], z[1][1]),
                            pack_bf16(z[1][2], z[1][3])};
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) {
      uint32_t r[4];
      ldsm_x4_t(r, sDZ + swz128(((mi & 1) << 3) + mr, 2 * qq + (mi >> 1)));
      const uint32_t b0[2] = {r[0], r[1]}, b1[2] = {r[2], r[3]};
      mma_bf16_16816(Hc[2 * qq], za, b0);
      mma_bf16_16816(Hc[2 * qq + 1], za, b1);
    }
    // Every register loaded from the stage is consumed: hand it back (the proxy fence
    // orders these reads before the refill's async-proxy write).
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  if (!ok) {
    if (lane == 0) {
      if (!*abort_flag) report_error(p.status, TTT_ERR_TIMEOUT, kWhereHmapConsumer, unit);
      *abort_flag = 1;
    }
    return;
  }

  // H_s [i][j] (row i: this warp's Phi column) and A_s = Phi at the segment's end.
  float* Hs = p.hA + (static_cast<size_t>(unit) * nseg + seg - 1) * 2 * kD * kD;
  float* As = Hs + kD * kD;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int n = 8 * q + 2 * tg;
    *reinterpret_cast<float2*>(Hs + (jw + g) * kD + n) = make_float2(Hc[q][0], Hc[q][1]);
    *reinterpret_cast<float2*>(Hs + (jw + g + 8) * kD + n) = make_float2(Hc[q][2], Hc[q][3]);
    As[n * kD + jw + g] = Pt[q][0];
    As[(n + 1) * kD + jw + g] = Pt[q][1];
    As[n * kD + jw + g + 8] = Pt[q][2];
    As[(n + 1) * kD + jw + g + 8] = Pt[q][3];
  }
}

constexpr int kRcCols = 8;
constexpr int kRcThreads = 128;

// G_end(S-1) = dW_out; G_end(s - 1) = A_s^T G_end(s) + H_s for s = S-1 .. 1, for this
// CTA's 8 columns of one unit.
__global__ void __launch_bounds__(kRcThreads) linear_bwd_rcombine_kernel(LinearBwdParams p) {
  __shared__ __align__(16) float sA[kD * kD];
  __shared__ __align__(16) float sG[kD * kRcCols];
  const int groups = kD / kRcCols;
  const int unit = blockIdx.x / groups;
  const int j0 = (blockIdx.x % groups) * kRcCols;
  const int nseg = p.bseg_count - 1;
  const int tid = threadIdx.x;
  const int i = tid >> 1;
  const int c = (tid & 1) * 4;
  *reinterpret_cast<float4*>(&sG[i * kRcCols + c]) =
      *reinterpret_cast<const float4*>(p.dW_out + static_cast<size_t>(unit) * kD * kD + i * kD + j0 + c);
  // A_s (8 float4 per thread) and this thread's four entries of H_s, fetched one step ahead.
  float4 ra[kD * kD / 4 / kRcThreads];
  float4 hv;
  auto fetch = [&](int s) {
    const float* Hs = p.hA + (static_cast<size_t>(unit) * nseg + s - 1) * 2 * kD * kD;
#pragma unroll
    for (int r = 0; r < kD * kD / 4 / kRcThreads; ++r)
      ra[r] = __ldcg(reinterpret_cast<const float4*>(Hs + kD * kD) + tid + kRcThreads * r);
    hv = __ldcg(reinterpret_cast<const float4*>(Hs + i * kD + j0 + c));
  };
  if (nseg >= 1) fetch(nseg);
  for (int s = nseg; s >= 1; --s) {
#pragma unroll
    for (int r = 0; r < kD * kD / 4 / kRcThreads; ++r) reinterpret_cast<float4*>(sA)[tid + kRcThreads * r] = ra[r];
    const float4 h4 = hv;
    __syncthreads();  // sA holds A_s; sG holds G_end(s)
    if (s > 1) fetch(s - 1);
    float acc[4] = {h4.x, h4.y, h4.z, h4.w};
    for (int k = 0; k < kD; ++k) {
      const float a = sA[k * kD + i];  // (A_s^T)[i][k]
      const float4 gv = *reinterpret_cast<const float4*>(&sG[k * kRcCols + c]);
      acc[0] = fmaf(a, gv.x, acc[0]);
      acc[1] = fmaf(a, gv.y, acc[1]);
      acc[2] = fmaf(a, gv.z, acc[2]);
      acc[3] = fmaf(a, gv.w, acc[3]);
    }
    __syncthreads();  // every thread is done reading sA and sG
    const float4 nv = make_float4(acc[0], acc[1], acc[2], acc[3]);
    *reinterpret_cast<float4*>(&sG[i * kRcCols + c]) = nv;
    *reinterpret_cast<float4*>(p.g_ends + (static_cast<size_t>(unit) * nseg + s - 1) * kD * kD + i * kD + j0 + c) = nv;
  }
}

}  // namespace

int linear_bwd_hmap_rows() { return kTile; }

cudaError_t launch_linear_bwd_hmap(const LinearBwdParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                                   const CUtensorMap& mdz, cudaStream_t stream) {
  if (p.units == 0 || p.bseg_count < 2) return cudaSuccess;
  linear_bwd_hmap_kernel<<<p.units * (p.bseg_count - 1), kThreads, kSmemBytes, stream>>>(mq, mk, mdz, p);
  return cudaGetLastError();
}

cudaError_t launch_linear_bwd_rcombine(const LinearBwdParams& p, cudaStream_t stream) {
  if (p.units == 0 || p.bseg_count < 2) return cudaSuccess;
  linear_bwd_rcombine_kernel<<<p.units * (kD / kRcCols), kRcThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace ttt
