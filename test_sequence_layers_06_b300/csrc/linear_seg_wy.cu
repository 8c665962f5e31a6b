// Segment affine maps of TTT-Linear on the tcgen05 tensor cores, 64 tokens per
// step (bf16 inputs, d = 64; b = 16, 32 or a multiple of 64).
//
// What is computed is the same as linear_seg_affine_kernel (linear_seg.cu): for a
// segment of whole chunks, the composed affine map X = [A | B] of its chunk
// updates, run on the 64 x 128 state X from [I | 0] with value rows [0 | V].
//
// Super-chunks. Take 64 consecutive tokens holding whole chunks (b = 16 or 32),
// X0 the state before them. Chunk c's error is taken at its own start state
// X0 - eta sum_{c' < c} K_c'^T E_c', so
//   E_c = K_c X0 - [0|V]_c - eta sum_{c' < c} (K_c K_c'^T) E_c',
// i.e. (I + eta N) E = R with R = K X0 - [0|V] and N the strictly block-lower
// part (chunk blocks) of K K^T. With T = (I + eta N)^-1:
//   X_end = X0 - eta K^T T R = X0 - eta Kh^T R,   Kh = T^T K.
// This is exact algebra on the chunk rule ("5 · TestingTime 训练与长上下文",
// sections 1.1 and 4); the pages do not write it. Kh depends only on the
// inputs, so two helper warps compute it ahead of time with warp-level MMAs,
// in registers: the 16 x 16 blocks of T^T by the short recurrence
// U_cr = -eta sum_m U_cm G_mr (U = T^T, G = K K^T blocks, U_cc = I), then
// Kh_c = K_c + sum_{r > c} U_cr K_r. They also store V transposed, so that the
// thread owning column j of B reads its 64 values with eight 16-byte loads.
// The chain that depends on X is two tensor-core products per 64 tokens
// instead of two per chunk:
//   R^T = X0^T K^T                    (M 128, N 64, K 64)
//   -eta R^T + eta [0|V]^T            (registers: thread r owns row r of X^T)
//   X^T += (-eta R^T) Kh              (M 128, N 64, K 64; Kh read MN-major)
// For b >= 64 every 64-token step lies inside one chunk: T = I, Kh = K, and X0
// stays the chunk-start state until the chunk ends.
//
// Roles (224 threads): warps 0-3 own the 128 rows of X^T (tensor memory <->
// registers <-> shared memory); warp 4 lane 0 issues the TMA loads and the
// MMAs; warps 5 and 6 compute Kh and V^T for even and odd steps. Every wait is
// bounded in time and gives up early when another role has given up.
#include "ttt_device.cuh"
#include "tcgen05.cuh"
#include "kernels.h"

namespace ttt {
namespace {

constexpr int kD = 64;
constexpr int kStep = 64;                         // tokens per super-chunk
constexpr int kStages = 3;
constexpr int kThreads = 224;
constexpr int kTileBytes = kStep * kD * 2;        // 8 KB: one 64 x 64 bf16 tile
constexpr int kXOff = 0;                          // X0^T bf16 [128][64] (and -eta E^T when b < 64)
constexpr int kPOff = 16384;                      // Kh[2] (b < 64) or -eta R^T (b >= 64); then V^T[2]
constexpr int kStageOff = kPOff + 4 * kTileBytes; // stages: K tile, V tile
constexpr int kBarOff = kStageOff + kStages * 2 * kTileBytes;
constexpr int kNumBars = 2 * kStages + 4 + 5;
constexpr int kMiscOff = kBarOff + kNumBars * 8;
constexpr int kSmemBytes = kMiscOff + 16 + 1024;  // + slack to align the base to 1024
constexpr uint32_t kCols = 128;                   // X^T: [0, 64); R^T: [64, 128)
constexpr uint32_t kIdR = tc::idesc_bf16_f32(128, 64, false, false);
constexpr uint32_t kIdU = tc::idesc_bf16_f32(128, 64, false, true);

enum : int { kWhereControl = 8, kWhereRows = 9, kWherePrep = 10, kWhereDrain = 11 };

// Whether block pair (r, m), m < r, of the step's four 16-token blocks lies in
// different chunks (chunks of bt tokens): only then does G_rm enter N.
__device__ __forceinline__ bool needed(int r, int m, int bt) { return m < r && (16 * m) / bt < (16 * r) / bt; }

// Kh = T^T K for one 64-token step (b = 16 or 32), written as rows of tokens
// (128-byte swizzled), the MN-major B operand of the state update.
__device__ void prep_khat(uint32_t sK, uint8_t* kh, float neta, int bt, int lane) {
  const int g = lane >> 2;
  const int tg = lane & 3;
  const int mi = lane >> 3;
  const int mr = lane & 7;
  // G_rm = K_r K_m^T for r > m, kept as B fragments of G_mr = G_rm^T
  // (k = tokens of block m, n = tokens of block r; two 8-wide n-tiles).
  uint32_t gb[4][4][2][2];
#pragma unroll
  for (int r = 1; r < 4; ++r)
#pragma unroll
    for (int m = 0; m < 3; ++m) {
      if (!needed(r, m, bt)) continue;
      float acc[2][4] = {};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t a[4], bb[4];
        ldsm_x4(a, sK + swz128(16 * r + ((mi & 1) << 3) + mr, 2 * k + (mi >> 1)));
        ldsm_x4(bb, sK + swz128(16 * m + ((mi >> 1) << 3) + mr, 2 * k + (mi & 1)));
        const uint32_t b0[2] = {bb[0], bb[1]}, b1[2] = {bb[2], bb[3]};
        mma_bf16_16816(acc[0], a, b0);
        mma_bf16_16816(acc[1], a, b1);
      }
#pragma unroll
      for (int nr = 0; nr < 2; ++nr) {
        gb[r][m][nr][0] = pack_bf16(acc[0][2 * nr], acc[0][2 * nr + 1]);
        gb[r][m][nr][1] = pack_bf16(acc[1][2 * nr], acc[1][2 * nr + 1]);
      }
    }
  // U = T^T by blocks, as A fragments (rows: tokens of block c, k: tokens of block r).
  const uint32_t eye = (g == 2 * tg ? 0x00003F80u : 0u) | (g == 2 * tg + 1 ? 0x3F800000u : 0u);
  const uint32_t ident[4] = {eye, 0u, 0u, eye};
  uint32_t ua[4][4][4];
  bool nz[4][4];
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int r = 0; r < 4; ++r) nz[c][r] = false;
#pragma unroll
  for (int dist = 1; dist < 4; ++dist)
#pragma unroll
    for (int c = 0; c + dist < 4; ++c) {
      const int r = c + dist;
      float acc[2][4] = {};
      bool any = false;
#pragma unroll
      for (int m = c; m < r; ++m) {
        if (!needed(r, m, bt) || (m > c && !nz[c][m])) continue;
        any = true;
        const uint32_t* a = m == c ? ident : ua[c][m];
        mma_bf16_16816(acc[0], a, gb[r][m][0]);
        mma_bf16_16816(acc[1], a, gb[r][m][1]);
      }
      nz[c][r] = any;
      ua[c][r][0] = pack_bf16(neta * acc[0][0], neta * acc[0][1]);
      ua[c][r][1] = pack_bf16(neta * acc[0][2], neta * acc[0][3]);
      ua[c][r][2] = pack_bf16(neta * acc[1][0], neta * acc[1][1]);
      ua[c][r][3] = pack_bf16(neta * acc[1][2], neta * acc[1][3]);
    }
  // Kh_c = K_c + sum_{r > c} U_cr K_r.
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    float acc[8][4];
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) {
      uint32_t a[4];
      ldsm_x4(a, sK + swz128(16 * c + ((mi & 1) << 3) + mr, 2 * qq + (mi >> 1)));
      acc[2 * qq][0] = bf16_lo(a[0]);
      acc[2 * qq][1] = bf16_hi(a[0]);
      acc[2 * qq][2] = bf16_lo(a[1]);
      acc[2 * qq][3] = bf16_hi(a[1]);
      acc[2 * qq + 1][0] = bf16_lo(a[2]);
      acc[2 * qq + 1][1] = bf16_hi(a[2]);
      acc[2 * qq + 1][2] = bf16_lo(a[3]);
      acc[2 * qq + 1][3] = bf16_hi(a[3]);
    }
#pragma unroll
    for (int r = c + 1; r < 4; ++r) {
      if (!nz[c][r]) continue;
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        uint32_t bb[4];
        ldsm_x4_t(bb, sK + swz128(16 * r + ((mi & 1) << 3) + mr, 2 * qq + (mi >> 1)));
        const uint32_t b0[2] = {bb[0], bb[1]}, b1[2] = {bb[2], bb[3]};
        mma_bf16_16816(acc[2 * qq], ua[c][r], b0);
        mma_bf16_16816(acc[2 * qq + 1], ua[c][r], b1);
      }
    }
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      *reinterpret_cast<uint32_t*>(kh + swz128(16 * c + g, nt) + 4 * tg) = pack_bf16(acc[nt][0], acc[nt][1]);
      *reinterpret_cast<uint32_t*>(kh + swz128(16 * c + g + 8, nt) + 4 * tg) = pack_bf16(acc[nt][2], acc[nt][3]);
    }
  }
}

// V transposed into rows of value columns (128-byte swizzled).
__device__ void transpose_v(uint32_t sV, uint8_t* vtt, int lane) {
  const int mi = lane >> 3;
  const int mr = lane & 7;
  const uint32_t svt = smem_u32(vtt);
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) {
      uint32_t a[4];
      ldsm_x4(a, sV + swz128(16 * r + ((mi & 1) << 3) + mr, 2 * qq + (mi >> 1)));
      stsm_x4_t(svt + swz128(8 * (2 * qq + (mi >> 1)) + mr, 2 * r + (mi & 1)), a);
    }
  __syncwarp();
}

__global__ void __launch_bounds__(kThreads, 2)
    linear_seg_affine_wy_kernel(const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                                LinearParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOff);  // [kStages] TMA data landed
  uint64_t* sfree = full + kStages;                               // [kStages] MMAs done with the stage
  uint64_t* prepready = sfree + kStages;                          // [2] Kh, V^T written
  uint64_t* pfree = prepready + 2;                                // [2] MMAs and rows done with Kh, V^T
  uint64_t* rdone = pfree + 2;
  uint64_t* eready = rdone + 1;
  uint64_t* udone = rdone + 2;
  uint64_t* xready = rdone + 3;
  uint64_t* drain = rdone + 4;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kMiscOff + 4);

  const int maps = p.seg_count - 1;
  const int unit = blockIdx.x / maps;
  const int seg = blockIdx.x % maps;
  const int h = unit % p.H;
  const int t0 = seg * p.seg_len;
  const int n = p.seg_len / kStep;
  const bool wy = p.b < kStep;                   // b = 16 or 32: Kh differs from K
  const int spc = wy ? 1 : p.b / kStep;          // steps per chunk
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const float neta = -p.eta[h];

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&sfree[s], 1);
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(&prepready[q], 1);
      mbar_init(&pfree[q], 1);
    }
    mbar_init(rdone, 1);
    mbar_init(eready, 4);
    mbar_init(udone, 1);
    mbar_init(xready, 4);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(tslot, kCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;
  const uint32_t tX = tmem;
  const uint32_t tR = tmem + 64;
  uint8_t* sXp = smem + kXOff;
  uint8_t* sEp = wy ? smem + kXOff : smem + kPOff;
  auto stageK = [&](int s) { return smem + kStageOff + s * 2 * kTileBytes; };
  auto khp = [&](int q) { return smem + kPOff + q * kTileBytes; };        // Kh
  auto vtp = [&](int q) { return smem + kPOff + (2 + q) * kTileBytes; };  // V^T

  if (warp == 4) {
    // -------------------------------------------------- control: TMA and MMA issue
    if (lane == 0) {
      prefetch_tmap(&mk);
      prefetch_tmap(&mv);
      int loaded = 0;
      auto load = [&](int j) {
        const int s = j % kStages;
        mbar_arrive_expect_tx(&full[s], 2 * kTileBytes);
        tma_load_3d(stageK(s), &mk, &full[s], 0, t0 + j * kStep, unit);
        tma_load_3d(stageK(s) + kTileBytes, &mv, &full[s], 0, t0 + j * kStep, unit);
        loaded = j + 1;
      };
      if (!p.inject_stall)
        for (int j = 0; j < min(kStages, n); ++j) load(j);
      bool ok = true;
      int consumed = 0;  // steps whose TMA data this thread has seen land
      for (int j = 0; j < n; ++j) {
        const int s = j % kStages;
        const int q = j & 1;
        ok = mbar_wait_or_abort(&full[s], (j / kStages) & 1, p.timeout_ns, abort_flag);
        if (ok) consumed = j + 1;
        if (ok && j % spc == 0) ok = mbar_wait_or_abort(xready, (j / spc) & 1, p.timeout_ns, abort_flag);
        if (!ok) break;
        tc::fence_after_sync();
        const uint32_t sX = smem_u32(sXp);
        const uint32_t sB = smem_u32(stageK(s));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_bf16(tR, tc::sdesc(sX + 32 * kk, 16, 1024, tc::kSw128), tc::sdesc(sB + 32 * kk, 16, 1024, tc::kSw128),
                       kIdR, kk > 0 ? 1u : 0u);
        tc::commit(rdone);
        ok = mbar_wait_or_abort(eready, j & 1, p.timeout_ns, abort_flag);
        if (ok && wy) ok = mbar_wait_or_abort(&prepready[q], (j >> 1) & 1, p.timeout_ns, abort_flag);
        if (!ok) break;
        tc::fence_after_sync();
        const uint32_t sE = smem_u32(sEp);
        const uint32_t sK = smem_u32(wy ? khp(q) : stageK(s));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_bf16(tX, tc::sdesc(sE + 32 * kk, 16, 1024, tc::kSw128),
                       tc::sdesc(sK + 2048 * kk, 1024, 1024, tc::kSw128), kIdU, 1u);
        if (j % spc == spc - 1) tc::commit(udone);
        tc::commit(&pfree[q]);
        tc::commit(&sfree[s]);
        if (j + kStages < n && !p.inject_stall) {
          ok = mbar_wait_or_abort(&sfree[s], (j / kStages) & 1, p.timeout_ns, abort_flag);
          if (!ok) break;
          load(j + kStages);
        }
      }
      if (!ok) {
        if (!*abort_flag) report_error(p.status, TTT_ERR_TIMEOUT, kWhereControl, unit);
        *abort_flag = 1;
      }
      tc::commit(drain);
      if (!mbar_wait_bounded(drain, 0, p.timeout_ns)) report_error(p.status, TTT_ERR_TIMEOUT, kWhereDrain, unit);
      // Loads issued but not yet seen to land (each holds its own stage).
      for (int v = consumed; v < loaded; ++v)
        (void)mbar_wait_bounded(&full[v % kStages], (v / kStages) & 1, p.timeout_ns);
    }
  } else if (warp >= 5) {
    // -------------------------------------------------- Kh and V^T for every other step
    {
      bool ok = true;
      for (int j = warp - 5; j < n; j += 2) {
        const int s = j % kStages;
        const int q = j & 1;
        ok = mbar_wait_or_abort(&full[s], (j / kStages) & 1, p.timeout_ns, abort_flag);
        if (ok && j >= 2) ok = mbar_wait_or_abort(&pfree[q], ((j - 2) >> 1) & 1, p.timeout_ns, abort_flag);
        if (!ok) break;
        transpose_v(smem_u32(stageK(s) + kTileBytes), vtp(q), lane);
        if (wy) prep_khat(smem_u32(stageK(s)), khp(q), neta, p.b, lane);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&prepready[q]);
      }
      if (!ok && lane == 0) {
        if (!*abort_flag) report_error(p.status, TTT_ERR_TIMEOUT, kWherePrep, unit);
        *abort_flag = 1;
      }
    }
  } else {
    // -------------------------------------------------- rows of X^T
    const int r = threadIdx.x;  // 0..127
    const int half = r >> 6;    // 0: a column of A, 1: a column of B
    const int jc = r & 63;
    const uint32_t lanes = static_cast<uint32_t>(32 * warp) << 16;
    const int rx = (r >> 3) * 1024 + (r & 7) * 128;  // row r in a [128][64] 128-byte-swizzled tile

    {
      float v[16];
#pragma unroll
      for (int c = 0; c < 64; c += 16) {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = (half == 0 && c + i == jc) ? 1.f : 0.f;
        tc::st16(tX + lanes + c, v);
      }
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint32_t one = (half == 0 && (jc >> 3) == c) ? ((jc & 1) ? 0x3F800000u : 0x00003F80u) : 0u;
        const int slot = (jc & 7) >> 1;
        *reinterpret_cast<uint4*>(sXp + rx + (((c ^ (r & 7)) & 7) << 4)) =
            make_uint4(slot == 0 ? one : 0u, slot == 1 ? one : 0u, slot == 2 ? one : 0u, slot == 3 ? one : 0u);
      }
    }
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(xready);

    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int q = j & 1;
      if (!mbar_wait_or_abort(rdone, j & 1, p.timeout_ns, abort_flag)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      float v[64];
      tc::ld32(tR + lanes, v);
      tc::ld32(tR + lanes + 32, v + 32);
      if (half) {
        // Row jc of V^T, written by a helper warp: wait for it directly.
        if (!mbar_wait_or_abort(&prepready[q], (j >> 1) & 1, p.timeout_ns, abort_flag)) {
          ok = false;
          break;
        }
        const uint8_t* vrow = vtp(q) + jc * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 w = *reinterpret_cast<const uint4*>(vrow + (((c ^ (jc & 7)) & 7) << 4));
          const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            v[8 * c + 2 * e] -= bf16_lo(ww[e]);
            v[8 * c + 2 * e + 1] -= bf16_hi(ww[e]);
          }
        }
      }
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(sEp + rx + (((c ^ (r & 7)) & 7) << 4)) =
            make_uint4(pack_bf16(neta * v[8 * c], neta * v[8 * c + 1]), pack_bf16(neta * v[8 * c + 2], neta * v[8 * c + 3]),
                       pack_bf16(neta * v[8 * c + 4], neta * v[8 * c + 5]),
                       pack_bf16(neta * v[8 * c + 6], neta * v[8 * c + 7]));
      fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(eready);
      if (j % spc == spc - 1 && j + 1 < n) {
        if (!mbar_wait_or_abort(udone, (j / spc) & 1, p.timeout_ns, abort_flag)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        float x[64];
        tc::ld32(tX + lanes, x);
        tc::ld32(tX + lanes + 32, x + 32);
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(sXp + rx + (((c ^ (r & 7)) & 7) << 4)) =
              make_uint4(pack_bf16(x[8 * c], x[8 * c + 1]), pack_bf16(x[8 * c + 2], x[8 * c + 3]),
                         pack_bf16(x[8 * c + 4], x[8 * c + 5]), pack_bf16(x[8 * c + 6], x[8 * c + 7]));
        fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(xready);
      }
    }
    if (ok && mbar_wait_or_abort(udone, ((n - 1) / spc) & 1, p.timeout_ns, abort_flag)) {
      // (A_s or B_s)[i][jc] = X^T[r][i]
      tc::fence_after_sync();
      float* out = p.seg_maps + (static_cast<size_t>(unit) * maps + seg) * 2 * kD * kD + half * kD * kD;
      float x[64];
      tc::ld32(tX + lanes, x);
      tc::ld32(tX + lanes + 32, x + 32);
#pragma unroll
      for (int i = 0; i < 64; ++i) out[i * kD + jc] = x[i];
    } else {
      if (!*abort_flag) report_error(p.status, TTT_ERR_TIMEOUT, kWhereRows, unit);
      *abort_flag = 1;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kCols);
  }
}

}  // namespace

bool linear_seg_wy_supported(int b, int seg_len) {
  return b % 16 == 0 && (b % kStep == 0 || kStep % b == 0) && seg_len % kStep == 0 && seg_len % b == 0;
}

int linear_seg_wy_rows() { return kStep; }

cudaError_t launch_linear_seg_affine_wy(const LinearParams& p, const CUtensorMap& mk64, const CUtensorMap& mv64,
                                        cudaStream_t stream) {
  const int items = p.units * (p.seg_count - 1);
  if (items == 0) return cudaSuccess;
  static bool attr_set = false;  // idempotent; a race only repeats the call
  if (!attr_set) {
    const cudaError_t e =
        cudaFuncSetAttribute(linear_seg_affine_wy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  linear_seg_affine_wy_kernel<<<items, kThreads, kSmemBytes, stream>>>(mk64, mv64, p);
  return cudaGetLastError();
}

}  // namespace ttt
