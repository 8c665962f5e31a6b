// Segment-parallel form of the TTT-Linear scan (bf16 inputs, d = 64, b % 16 == 0).
//
// One chunk's gradient step ("5 · TestingTime 训练与长上下文", sections 1.1 and 4;
// "Test-Time Training (TTT) guide", section 3),
//   W <- W - eta K_c^T (K_c W - V_c),
// is affine in W: W <- A_c W + B_c with A_c = I - eta K_c^T K_c and
// B_c = eta K_c^T V_c. A run of chunks therefore maps its start state to its
// end state by the composition (A_s, B_s) of its chunks' maps. The pages do not
// write the update this way; it is exact algebra on it, and it lets one head's
// sequence be cut into S segments that run side by side:
//
//   1. linear_seg_affine_kernel (here, warp-level MMAs) or
//      linear_seg_affine_wy_kernel (linear_seg_wy.cu, tcgen05 tensor cores, the
//      default where it applies): (A_s, B_s) of every segment but the last, all
//      at once. It runs the chunk update on the 64 x 128 state X = [A | B] from
//      X = [I | 0]; the value rows are 0 for the A half and V_c for the B half,
//      so the A half follows A <- A_c A and the B half B <- A_c B + B_c.
//   2. linear_seg_combine_kernel: W_start(0) = W0 and
//      W_start(s + 1) = A_s W_start(s) + B_s, in fp32.
//   3. linear_mma_kernel on every segment from its start state: read-out of Z
//      and, for the last segment, the final state.
//
// The affine kernel uses the same register-resident scheme as linear_mma.cu:
// X^T lives in mma.sync accumulator fragments, each of 8 consumer warps owns 16
// of X's 128 columns, and a chunk larger than 16 tokens takes every tile's
// error at the chunk-start snapshot of X.
#include "ttt_device.cuh"
#include "kernels.h"


namespace ttt {
namespace {

constexpr int kD = 64;
constexpr int kTile = 16;
constexpr int kTileBytes = kTile * kD * 2;       // 2048
constexpr int kAffWarps = 8;                     // X = [A | B]: 8 groups of 16 columns
constexpr int kAffThreads = (kAffWarps + 1) * 32;
constexpr int kAffStages = 8;
constexpr int kAffStageBytes = 2 * kTileBytes;   // K and V tiles
constexpr int kAffBarOff = kAffStages * kAffStageBytes;
constexpr int kAffAbortOff = kAffBarOff + 2 * kAffStages * 8;
constexpr int kAffSmemBytes = kAffAbortOff + 16 + 1024;  // + slack to align the base to 1024
static_assert(kAffSmemBytes <= 48 * 1024, "fits the default dynamic shared memory limit");

enum : int { kWhereAffProducer = 3, kWhereAffConsumer = 4 };

__global__ void __launch_bounds__(kAffThreads, 2)
    linear_seg_affine_kernel(const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                             LinearParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kAffBarOff);
  uint64_t* empty = full + kAffStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAffAbortOff);

  const int maps = p.seg_count - 1;       // the last segment needs no map
  const int unit = blockIdx.x / p.seg_num;
  const int seg = p.seg_first + blockIdx.x % p.seg_num;
  const int h = unit % p.H;
  const int t0 = seg * p.seg_len;
  const int num_tiles = p.seg_len / kTile;  // segments with a map are full
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kAffStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kAffWarps);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kAffWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&mk);
      prefetch_tmap(&mv);
      int issued = 0;
      for (int u = 0; u < num_tiles; ++u) {
        const int s = u % kAffStages;
        if (u >= kAffStages && !mbar_wait_bounded(&empty[s], ((u / kAffStages) - 1) & 1, p.timeout_ns)) {
          report_error(p.status, TTT_ERR_TIMEOUT, kWhereAffProducer, unit);
          *abort_flag = 1;
          break;
        }
        if (*abort_flag || p.inject_stall) break;
        mbar_arrive_expect_tx(&full[s], kAffStageBytes);
        uint8_t* st = smem + s * kAffStageBytes;
        tma_load_3d(st, &mk, &full[s], 0, t0 + u * kTile, unit);
        tma_load_3d(st + kTileBytes, &mv, &full[s], 0, t0 + u * kTile, unit);
        ++issued;
      }
      for (int u = (issued > kAffStages ? issued - kAffStages : 0); u < issued; ++u)
        (void)mbar_wait_bounded(&full[u % kAffStages], (u / kAffStages) & 1, p.timeout_ns);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2;
  const int tg = lane & 3;
  const int mi = lane >> 3;
  const int mr = lane & 7;
  const int half = warp >> 2;     // 0: columns of A, 1: columns of B
  const int cw = warp & 3;        // which 16 columns of that half
  const int jw = 16 * cw;
  const float neta = -p.eta[h];

  // X^T fragments (rows j = jw + g, jw + g + 8; columns i = 8q + 2tg, +1).
  // A starts as the identity, B as zero.
  float Xt[8][4];
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int i = 8 * q + 2 * tg;
    const float one = half == 0 ? 1.f : 0.f;
    Xt[q][0] = (i == jw + g) ? one : 0.f;
    Xt[q][1] = (i + 1 == jw + g) ? one : 0.f;
    Xt[q][2] = (i == jw + g + 8) ? one : 0.f;
    Xt[q][3] = (i + 1 == jw + g + 8) ? one : 0.f;
  }
  uint32_t xa[4][4];  // bf16 A fragments of the chunk-start X^T

  for (int u = 0; u < num_tiles; ++u) {
    const int s = u % kAffStages;
    if (!mbar_wait_bounded(&full[s], (u / kAffStages) & 1, p.timeout_ns)) {
      report_error(p.status, TTT_ERR_TIMEOUT, kWhereAffConsumer, unit);
      *abort_flag = 1;
      break;
    }
    if (*abort_flag) break;
    const uint32_t sK = smem_u32(smem + s * kAffStageBytes);
    const uint32_t sV = sK + kTileBytes;

    if (((u * kTile) % p.b) == 0) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        xa[k][0] = pack_bf16(Xt[2 * k][0], Xt[2 * k][1]);
        xa[k][1] = pack_bf16(Xt[2 * k][2], Xt[2 * k][3]);
        xa[k][2] = pack_bf16(Xt[2 * k + 1][0], Xt[2 * k + 1][1]);
        xa[k][3] = pack_bf16(Xt[2 * k + 1][2], Xt[2 * k + 1][3]);
      }
    }

    // Accumulator of E^T = X_a^T K^T - [0 | V]^T: -V^T for the B half, 0 for the A half.
    float e[2][4], e2[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) e[nt][r] = e2[nt][r] = 0.f;
    if (half == 1) {
      uint32_t vt[4];
      ldsm_x4_t(vt, sV + swz128(((mi >> 1) << 3) + mr, 2 * cw + (mi & 1)));
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        e[nt][0] = -bf16_lo(vt[2 * nt]);
        e[nt][1] = -bf16_hi(vt[2 * nt]);
        e[nt][2] = -bf16_lo(vt[2 * nt + 1]);
        e[nt][3] = -bf16_hi(vt[2 * nt + 1]);
      }
    }

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
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) mma_bf16_16816(k < 2 ? e[nt] : e2[nt], xa[k], kb[nt][k]);

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
    uint32_t ea[4];
    ea[0] = pack_bf16(neta * (e[0][0] + e2[0][0]), neta * (e[0][1] + e2[0][1]));
    ea[1] = pack_bf16(neta * (e[0][2] + e2[0][2]), neta * (e[0][3] + e2[0][3]));
    ea[2] = pack_bf16(neta * (e[1][0] + e2[1][0]), neta * (e[1][1] + e2[1][1]));
    ea[3] = pack_bf16(neta * (e[1][2] + e2[1][2]), neta * (e[1][3] + e2[1][3]));
    // X^T += (-eta E^T) K: the chunk's gradient step on both halves.
#pragma unroll
    for (int q = 0; q < 8; ++q) mma_bf16_16816(Xt[q], ea, kbt[q]);
    // Release the stage only once every register loaded from it has been consumed
    // (no load from it outstanding); the proxy fence orders these generic-proxy
    // reads before the producer's async-proxy refill.
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }

  // (A_s or B_s)[i][j] = X^T[j][i].
  float* out = p.seg_maps + (static_cast<size_t>(unit) * maps + seg) * 2 * kD * kD + half * kD * kD;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int i = 8 * q + 2 * tg;
    out[i * kD + jw + g] = Xt[q][0];
    out[(i + 1) * kD + jw + g] = Xt[q][1];
    out[i * kD + jw + g + 8] = Xt[q][2];
    out[(i + 1) * kD + jw + g + 8] = Xt[q][3];
  }
}

// W_start(s + 1) = A_s W_start(s) + B_s for the maps s of the launch's range
// (seg_first ..), starting from W0 for the first segment,
// in fp32. The columns of W are independent, so a CTA serves 8 columns of one
// unit and a unit's 64 columns spread over 8 CTAs. Thread (i, c) holds row i,
// columns 4c .. 4c+3 of its CTA's slice.
constexpr int kCmbCols = 8;
constexpr int kCmbThreads = 128;
constexpr int kCmbPad = 68;   // row stride of A in shared memory (floats): conflict-free 16-byte reads
constexpr int kCmbRing = 4;   // maps in flight: the chain's loads run this many steps ahead

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__global__ void __launch_bounds__(kCmbThreads) linear_seg_combine_kernel(LinearParams p) {
  extern __shared__ __align__(16) float cmb_smem[];
  float* sA = cmb_smem;                            // [kCmbRing][kD][kCmbPad]
  float* sB = sA + kCmbRing * kD * kCmbPad;        // [kCmbRing][kCmbThreads][4]: this thread's entries of B
  float* sW = sB + kCmbRing * kCmbThreads * 4;     // [kD][kCmbCols]
  const int groups = kD / kCmbCols;
  const int unit = blockIdx.x / groups;
  const int j0 = (blockIdx.x % groups) * kCmbCols;
  const int h = unit % p.H;
  const int maps = p.seg_count - 1;
  const int tid = threadIdx.x;
  const int i = tid >> 1;
  const int c = (tid & 1) * 4;

  // W_start(seg_first): W0[h] for the first segment, else what the combine of the
  // previous maps wrote (this CTA's columns).
  const float* Ws = p.seg_first == 0
                        ? p.W0 + static_cast<size_t>(h) * kD * kD
                        : p.seg_starts + (static_cast<size_t>(unit) * maps + p.seg_first - 1) * kD * kD;
  *reinterpret_cast<float4*>(&sW[i * kCmbCols + c]) = __ldcg(reinterpret_cast<const float4*>(Ws + i * kD + j0 + c));

  // Map s into ring slot (s - seg_first) % kCmbRing: A (4096 floats, 8 x 16 bytes per thread)
  // and this thread's four entries of B, as one cp.async group.
  const int s_end = p.seg_first + p.seg_num;
  auto fetch = [&](int s) {
    const int slot = (s - p.seg_first) % kCmbRing;
    const float* A = p.seg_maps + (static_cast<size_t>(unit) * maps + s) * 2 * kD * kD;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int f = (tid + kCmbThreads * r) * 4;
      cp_async16(&sA[(slot * kD + f / kD) * kCmbPad + f % kD], A + f);
    }
    cp_async16(&sB[(slot * kCmbThreads + tid) * 4], A + kD * kD + i * kD + j0 + c);
  };
#pragma unroll
  for (int r = 0; r < kCmbRing; ++r) {
    if (p.seg_first + r < s_end) fetch(p.seg_first + r);
    cp_async_commit();  // one group per map (empty past the end), so the count below holds
  }
  for (int s = p.seg_first; s < s_end; ++s) {
    const int slot = (s - p.seg_first) % kCmbRing;
    cp_async_wait<kCmbRing - 1>();  // this thread's copies of map s have landed
    __syncthreads();                // everyone's have; sW holds W_start(s)
    const float* a_s = sA + slot * kD * kCmbPad;
    const float4 b = *reinterpret_cast<const float4*>(&sB[(slot * kCmbThreads + tid) * 4]);
    float acc[2][4] = {{b.x, b.y, b.z, b.w}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int k = 0; k < kD; k += 4) {
      const float4 a = *reinterpret_cast<const float4*>(&a_s[i * kCmbPad + k]);
      const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const float4 w = *reinterpret_cast<const float4*>(&sW[(k + kk) * kCmbCols + c]);
        float* o = acc[kk & 1];
        o[0] = fmaf(av[kk], w.x, o[0]);
        o[1] = fmaf(av[kk], w.y, o[1]);
        o[2] = fmaf(av[kk], w.z, o[2]);
        o[3] = fmaf(av[kk], w.w, o[3]);
      }
    }
    const float4 nw = make_float4(acc[0][0] + acc[1][0], acc[0][1] + acc[1][1], acc[0][2] + acc[1][2],
                                  acc[0][3] + acc[1][3]);
    __syncthreads();  // every thread is done reading sW and this slot
    *reinterpret_cast<float4*>(&sW[i * kCmbCols + c]) = nw;
    *reinterpret_cast<float4*>(p.seg_starts + (static_cast<size_t>(unit) * maps + s) * kD * kD + i * kD + j0 + c) =
        nw;
    if (s + kCmbRing < s_end) fetch(s + kCmbRing);  // refill the slot just read
    cp_async_commit();
  }
  cp_async_wait<0>();
}

}  // namespace

bool linear_seg_supported(const LinearParams& p) { return p.d == kD && p.b % kTile == 0 && p.bf16; }

cudaError_t launch_linear_seg_affine(const LinearParams& p, const CUtensorMap& mk, const CUtensorMap& mv,
                                     cudaStream_t stream) {
  const int items = p.units * p.seg_num;
  if (items == 0) return cudaSuccess;
  linear_seg_affine_kernel<<<items, kAffThreads, kAffSmemBytes, stream>>>(mk, mv, p);
  return cudaGetLastError();
}

cudaError_t launch_linear_seg_combine(const LinearParams& p, cudaStream_t stream) {
  if (p.seg_count < 2 || p.units == 0 || p.seg_num == 0) return cudaSuccess;
  constexpr int smem = (kCmbRing * kD * kCmbPad + kCmbRing * kCmbThreads * 4 + kD * kCmbCols) * 4;
  const cudaError_t e =
      cudaFuncSetAttribute(linear_seg_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  linear_seg_combine_kernel<<<p.units * (kD / kCmbCols), kCmbThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace ttt
