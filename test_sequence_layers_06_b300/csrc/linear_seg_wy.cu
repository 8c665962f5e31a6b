// Segment affine maps of TTT-Linear on the tcgen05 tensor cores, one product
// per 64 tokens on the serial chain (bf16 inputs, d = 64; b = 16, 32 or a
// multiple of 64).
//
// What is computed is the same as linear_seg_affine_kernel (linear_seg.cu): for a
// segment of whole chunks, the composed affine map X = [A | B] of its chunk
// updates, run on the 64 x 128 state X from [I | 0] with value rows [0 | V].
//
// Groups. A group is 64 tokens holding whole chunks (b = 16, 32, 64) or one
// whole chunk (b a multiple of 64). Chunk c's error is taken at its own start
// state, E_c = K_c X_c - [0|V]_c with X_c = X0 - eta sum_{c' < c} K_c'^T E_c',
// so (I + eta N) E = K X0 - [0|V] with N the strictly block-lower part (chunk
// blocks) of K K^T. With T = (I + eta N)^-1 and Kh = T^T K the group's update is
//   X_end = X0 - eta Kh^T (K X0 - [0|V]) = X0 + M X0 + [0 | Q],
//   M = -eta Kh^T K,   Q = eta Kh^T V,
// an affine map that depends on the inputs only (for b >= 64, Kh = K and the
// sums run over the chunk's 64-token steps). This is exact algebra on the chunk
// rule ("5 · TestingTime 训练与长上下文", sections 1.1 and 4); the pages do not
// write it. So the serial chain is one tensor-core product per group,
//   X^T += X^T M^T                     (M 128, N 64, K 64; A in tensor memory),
// then the row threads add Q^T to the B rows of X^T (fp32) and round the new
// X^T to bf16 (the next product's A operand). Everything else runs ahead of it:
//   - three helper warps form Kh = T^T K with warp-level MMAs, in registers, each
//     for every third step: the 16 x 16 blocks of T^T by
//     U_cr = -eta sum_m U_cm G_mr (G = K K^T blocks, U_cc = I), then
//     Kh_c = K_c + sum_{r > c} U_cr K_r;
//   - one M = 128 product [K^T; V^T] Kh = [-M^T / eta; Q^T / eta] per step, two
//     groups ahead, into one of two tensor-memory buffers;
//   - while the chain product of the previous group runs, the A-row threads
//     round the top half to bf16 M^T (the chain's B operand, read MN-major: no
//     transposition anywhere) and the B-row threads take their row of Q^T
//     into registers (bf16 pairs, the rounding Q^T would get as an operand).
// Products run in issue order, so the control lane issues a group's prep product
// only after the previous chain product has landed: it then fills the pipe while
// the rows refresh X^T, instead of delaying that chain product.
//
// Roles (256 threads): warps 0-3 own the 128 rows of X^T and of the prep
// product; warp 4 lane 0 issues the TMA loads and the MMAs; warps 5-7 compute
// Kh for every third step, each into its own buffer. Every wait is bounded in
// time and gives up early when another role has given up.
#include "ttt_device.cuh"
#include "tcgen05.cuh"
#include "kernels.h"

namespace ttt {
namespace {

constexpr int kD = 64;
constexpr int kStep = 64;                          // tokens per TMA step
constexpr int kStages = 4;                         // K, V stages (a split K ring measured slower)
constexpr int kHelpers = 3;                        // Kh warps (b < 64), one buffer each
constexpr int kThreads = (5 + kHelpers) * 32;
constexpr int kTileBytes = kStep * kD * 2;         // 8 KB: one 64 x 64 bf16 tile
constexpr int kMOff = 0;                           // [2] M^T tiles, bf16 [64][64]
constexpr int kStageOff = kMOff + 2 * kTileBytes;  // [kStages] x (K tile, V tile)
constexpr int kKhOff = kStageOff + kStages * 2 * kTileBytes;  // Kh [kHelpers] (b < 64)
constexpr int kBarOff = kKhOff + kHelpers * kTileBytes;
constexpr int kNumBars = 2 * kStages + kHelpers + 2 + 2 + 2 + 3;
static_assert(kNumBars * 8 + 16 + 1024 + kBarOff <= 113 * 1024 - 512, "two CTAs per SM");
constexpr int kMiscOff = kBarOff + kNumBars * 8;     // TMEM address, abort flag, steps loaded
constexpr int kSmemBytes = kMiscOff + 16 + 1024;   // + slack to align the base to 1024
// Tensor memory: X^T fp32 [0, 64); prep [2] x 64 at [64, 192); X^T bf16 [192, 224).
constexpr uint32_t kCols = 256;
constexpr uint32_t kIdChain = tc::idesc_bf16_f32(128, 64, false, true);  // A from tensor memory
constexpr uint32_t kIdPrep = tc::idesc_bf16_f32(128, 64, true, true);

enum : int { kWhereControl = 8, kWhereRows = 9, kWherePrep = 10, kWhereDrain = 11 };

// Whether block pair (r, m), m < r, of a step's four 16-token blocks lies in
// different chunks (chunks of bt tokens): only then does G_rm enter N.
__device__ __forceinline__ bool needed(int r, int m, int bt) { return m < r && (16 * m) / bt < (16 * r) / bt; }

// The 16 x 16 blocks of U = T^T for one 64-token step (b = 16 or 32), as bf16 A
// fragments (rows: tokens of block c, k: tokens of block r), and which are nonzero.
__device__ void prep_u(uint32_t sK, float neta, int bt, int lane, uint32_t (&ua)[4][4][4], bool (&nz)[4][4]) {
  const int g = lane >> 2;
  const int tg = lane & 3;
  const int mi = lane >> 3;
  const int mr = lane & 7;
  // G_rm = K_r K_m^T for r > m, kept as B fragments of G_mr = G_rm^T
  // (k = tokens of block m, n = tokens of block r; two 8-wide n-tiles). Each
  // k-step loads every block's fragments once and feeds all the pairs.
  float gacc[4][4][2][4];
#pragma unroll
  for (int r = 1; r < 4; ++r)
#pragma unroll
    for (int m = 0; m < 3; ++m)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) gacc[r][m][nt][e] = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t a[4][4], bb[4][4];
#pragma unroll
    for (int r = 1; r < 4; ++r)
      if (needed(r, 0, bt) || needed(r, r - 1, bt))
        ldsm_x4(a[r], sK + swz128(16 * r + ((mi & 1) << 3) + mr, 2 * k + (mi >> 1)));
#pragma unroll
    for (int m = 0; m < 3; ++m)
      if (needed(3, m, bt) || needed(m + 1, m, bt))
        ldsm_x4(bb[m], sK + swz128(16 * m + ((mi >> 1) << 3) + mr, 2 * k + (mi & 1)));
#pragma unroll
    for (int r = 1; r < 4; ++r)
#pragma unroll
      for (int m = 0; m < 3; ++m) {
        if (!needed(r, m, bt)) continue;
        const uint32_t b0[2] = {bb[m][0], bb[m][1]}, b1[2] = {bb[m][2], bb[m][3]};
        mma_bf16_16816(gacc[r][m][0], a[r], b0);
        mma_bf16_16816(gacc[r][m][1], a[r], b1);
      }
  }
  uint32_t gb[4][4][2][2];
#pragma unroll
  for (int r = 1; r < 4; ++r)
#pragma unroll
    for (int m = 0; m < 3; ++m) {
      if (!needed(r, m, bt)) continue;
#pragma unroll
      for (int nr = 0; nr < 2; ++nr) {
        gb[r][m][nr][0] = pack_bf16(gacc[r][m][0][2 * nr], gacc[r][m][0][2 * nr + 1]);
        gb[r][m][nr][1] = pack_bf16(gacc[r][m][1][2 * nr], gacc[r][m][1][2 * nr + 1]);
      }
    }
  const uint32_t eye = (g == 2 * tg ? 0x00003F80u : 0u) | (g == 2 * tg + 1 ? 0x3F800000u : 0u);
  const uint32_t ident[4] = {eye, 0u, 0u, eye};
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
}

// Kh_c = K_c + sum_{r > c} U_cr K_r, written as rows of tokens (128-byte swizzled).
__device__ void prep_kh(uint32_t sK, uint8_t* kh, int lane, const uint32_t (&ua)[4][4][4], const bool (&nz)[4][4]) {
  const int mi = lane >> 3;
  const int mr = lane & 7;
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
    // Rows 16c.., columns 16qq..: the accumulator fragments are stmatrix's
    // register layout (matrices: rows 0-7 / 8-15 x columns 0-7 / 8-15).
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) {
      const uint32_t v[4] = {pack_bf16(acc[2 * qq][0], acc[2 * qq][1]), pack_bf16(acc[2 * qq][2], acc[2 * qq][3]),
                             pack_bf16(acc[2 * qq + 1][0], acc[2 * qq + 1][1]),
                             pack_bf16(acc[2 * qq + 1][2], acc[2 * qq + 1][3])};
      stsm_x4(smem_u32(kh) + swz128(16 * c + ((mi & 1) << 3) + mr, 2 * qq + (mi >> 1)), v);
    }
  }
}

__global__ void __launch_bounds__(kThreads, 2)
    linear_seg_affine_wy_kernel(const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                                LinearParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOff);  // [kStages] TMA data landed
  uint64_t* sfree = full + kStages;                               // [kStages] the step's product is done
  uint64_t* khready = sfree + kStages;                            // [kHelpers] Kh of step j in buffer j % kHelpers
  uint64_t* pdone = khready + kHelpers;  // [2] the group's prep product is in its tensor-memory buffer
  uint64_t* mqready = pdone + 2;      // [2] bf16 M^T written to buffer g & 1 (2 warp arrivals)
  uint64_t* qtaken = pdone + 4;       // [2] Q^T of buffer g & 1 read into registers (2 warp arrivals)
  uint64_t* xready = pdone + 6;       // X^T refreshed (4 warp arrivals)
  uint64_t* xdone = pdone + 7;        // the group's chain product is done
  uint64_t* drain = pdone + 8;        // every MMA issued has completed
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kMiscOff + 4);
  // Steps whose TMA load the control lane has issued. A stage is reloaded only
  // after the product of its previous step, so once this passes j the stage
  // barrier is in step j's phase: the helpers read it before they wait on that
  // barrier by parity (they run ahead and could otherwise see the phase before).
  int* n_loaded = reinterpret_cast<int*>(smem + kMiscOff + 8);

  const int maps = p.seg_count - 1;
  const int unit = blockIdx.x / p.seg_num;
  const int seg = p.seg_first + blockIdx.x % p.seg_num;
  const int h = unit % p.H;
  const int t0 = seg * p.seg_len;
  const int n = p.seg_len / kStep;                // TMA steps
  const bool wy = p.b < kStep;                    // b = 16 or 32: Kh differs from K
  const int spc = wy ? 1 : p.b / kStep;           // steps per group
  const int ng = n / spc;                         // groups
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const float eta = p.eta[h];

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&sfree[s], 1);
    }
    for (int q = 0; q < kHelpers; ++q) mbar_init(&khready[q], 1);
    mbar_init(&pdone[0], 1);
    mbar_init(&pdone[1], 1);
    mbar_init(&mqready[0], 2);
    mbar_init(&mqready[1], 2);
    mbar_init(&qtaken[0], 2);
    mbar_init(&qtaken[1], 2);
    mbar_init(xready, 4);
    mbar_init(xdone, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    *n_loaded = 0;
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
  const uint32_t tP = tmem + 64;  // + 64 * (group & 1)
  const uint32_t tXb = tmem + 192;
  auto stageK = [&](int s) { return smem + kStageOff + s * 2 * kTileBytes; };
  auto mtile = [&](int q) { return smem + kMOff + q * kTileBytes; };
  auto khp = [&](int q) { return smem + kKhOff + q * kTileBytes; };

  if (warp == 4) {
    // -------------------------------------------------- control: TMA and MMA issue
    if (lane == 0) {
      prefetch_tmap(&mk);
      prefetch_tmap(&mv);
      int loaded = 0, consumed = 0;
      auto load = [&](int j) {
        const int s = j % kStages;
        mbar_arrive_expect_tx(&full[s], 2 * kTileBytes);
        tma_load_3d(stageK(s), &mk, &full[s], 0, t0 + j * kStep, unit);
        tma_load_3d(stageK(s) + kTileBytes, &mv, &full[s], 0, t0 + j * kStep, unit);
        loaded = j + 1;
        st_release(n_loaded, loaded);
      };
      if (!p.inject_stall)
        for (int j = 0; j < min(kStages, n); ++j) load(j);
      // [K^T; V^T] Kh of group g, accumulated over its steps into buffer g & 1.
      auto issue_prep = [&](int g) -> bool {
        const uint32_t dst = tP + 64 * (g & 1);
        for (int j = g * spc; j < (g + 1) * spc; ++j) {
          const int s = j % kStages;
          if (j >= 1 && j + kStages - 1 < n && !p.inject_stall) {  // refill the stage of step j-1
            if (!mbar_wait_or_abort(&sfree[(j - 1) % kStages], ((j - 1) / kStages) & 1, p.timeout_ns, abort_flag))
              return false;
            load(j + kStages - 1);
          }
          // b < 64: the helper saw step j's tiles land before it raised khready, so
          // khready alone orders these products after the TMA writes.
          if (wy) {
            if (!mbar_wait_or_abort(&khready[j % kHelpers], (j / kHelpers) & 1, p.timeout_ns, abort_flag))
              return false;
          } else if (!mbar_wait_or_abort(&full[s], (j / kStages) & 1, p.timeout_ns, abort_flag)) {
            return false;
          }
          consumed = j + 1;
          tc::fence_after_sync();
          const uint32_t sK = smem_u32(stageK(s));
          const uint32_t sB = wy ? smem_u32(khp(j % kHelpers)) : sK;
          const bool first = (j % spc) == 0;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // A: K tile then V tile, MN-major, 8 KB apart; B: Kh, MN-major
            tc::mma_bf16(dst, tc::sdesc(sK + 2048 * kk, kTileBytes, 1024, tc::kSw128),
                         tc::sdesc(sB + 2048 * kk, 1024, 1024, tc::kSw128), kIdPrep, (!first || kk > 0) ? 1u : 0u);
          tc::commit(&sfree[s]);
        }
        tc::commit(&pdone[g & 1]);
        return true;
      };
      bool ok = issue_prep(0);
      if (ok && ng > 1) ok = issue_prep(1);
      for (int g = 0; ok && g < ng; ++g) {
        ok = mbar_wait_or_abort(&mqready[g & 1], (g >> 1) & 1, p.timeout_ns, abort_flag) &&
             mbar_wait_or_abort(xready, g & 1, p.timeout_ns, abort_flag);
        if (!ok) break;
        tc::fence_after_sync();
        const uint32_t sM = smem_u32(mtile(g & 1));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_bf16_ta(tX, tXb + 8 * kk, tc::sdesc(sM + 2048 * kk, 1024, 1024, tc::kSw128), kIdChain, 1u);
        tc::commit(xdone);
        // Let the chain product land before anything else enters the pipe; the
        // prep buffer of group g is free once its Q^T rows have been read.
        ok = mbar_wait_or_abort(xdone, g & 1, p.timeout_ns, abort_flag) &&
             mbar_wait_or_abort(&qtaken[g & 1], (g >> 1) & 1, p.timeout_ns, abort_flag);
        if (ok && g + 2 < ng) ok = issue_prep(g + 2);
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
    // -------------------------------------------------- Kh for every kHelpers-th step
    if (wy) {
      bool ok = true;
      for (int j = warp - 5; j < n; j += kHelpers) {
        const int s = j % kStages;
        ok = __all_sync(0xffffffffu, wait_count_or_abort(n_loaded, j + 1, p.timeout_ns, abort_flag) &&
                                         mbar_wait_or_abort(&full[s], (j / kStages) & 1, p.timeout_ns,
                                                            abort_flag));
        if (!ok) break;
        uint32_t ua[4][4][4];
        bool nz[4][4];
        prep_u(smem_u32(stageK(s)), -eta, p.b, lane, ua, nz);
        // The Kh buffer's previous user, step j - kHelpers, must have finished its product.
        const int jp = j - kHelpers;
        if (jp >= 0) ok = mbar_wait_or_abort(&sfree[jp % kStages], (jp / kStages) & 1, p.timeout_ns, abort_flag);
        if (!ok) break;
        prep_kh(smem_u32(stageK(s)), khp(j % kHelpers), lane, ua, nz);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&khready[j % kHelpers]);
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

    // X^T = [I | 0]^T in fp32 and as a bf16 A operand (two bf16 per column, the
    // even k in the low half).
    {
      float v[16];
#pragma unroll
      for (int c = 0; c < 64; c += 16) {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = (half == 0 && c + i == jc) ? 1.f : 0.f;
        tc::st16(tX + lanes + c, v);
      }
      uint32_t xb[32];
#pragma unroll
      for (int c = 0; c < 32; ++c)
        xb[c] = (half == 0 && (jc >> 1) == c) ? ((jc & 1) ? 0x3F800000u : 0x00003F80u) : 0u;
      tc::st32(tXb + lanes, xb);
    }
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(xready);

    // Group g's prep product: the A rows (warps 0, 1) write bf16 M^T = -eta x
    // (row r of the top half) for the chain; the B rows (warps 2, 3) keep
    // Q^T = eta x (row r of the bottom half) as bf16 pairs in qv.
    uint8_t* mrow = smem + kMOff + ((jc >> 3) * 1024 + (jc & 7) * 128);
    uint32_t qv[32];
    auto convert = [&](int g) -> bool {
      if (!mbar_wait_or_abort(&pdone[g & 1], (g >> 1) & 1, p.timeout_ns, abort_flag)) return false;
      tc::fence_after_sync();
      if (half == 0) {
        uint8_t* dst = mrow + (g & 1) * kTileBytes;
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          float v[32];
          tc::ld32(tP + 64 * (g & 1) + lanes + 32 * part, v);
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            const int c = 4 * part + cc;
            *reinterpret_cast<uint4*>(dst + (((c ^ (jc & 7)) & 7) << 4)) =
                make_uint4(pack_bf16(-eta * v[8 * cc], -eta * v[8 * cc + 1]),
                           pack_bf16(-eta * v[8 * cc + 2], -eta * v[8 * cc + 3]),
                           pack_bf16(-eta * v[8 * cc + 4], -eta * v[8 * cc + 5]),
                           pack_bf16(-eta * v[8 * cc + 6], -eta * v[8 * cc + 7]));
          }
        }
        fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&mqready[g & 1]);
      } else {
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          float v[32];
          tc::ld32(tP + 64 * (g & 1) + lanes + 32 * part, v);
#pragma unroll
          for (int c = 0; c < 16; ++c) qv[16 * part + c] = pack_bf16(eta * v[2 * c], eta * v[2 * c + 1]);
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&qtaken[g & 1]);
      }
      return true;
    };

    bool ok = convert(0);
    for (int g = 0; ok && g < ng; ++g) {
      if (half == 0 && g + 1 < ng && !(ok = convert(g + 1))) break;
      if (!(ok = mbar_wait_or_abort(xdone, g & 1, p.timeout_ns, abort_flag))) break;
      tc::fence_after_sync();
      float x[64];
      tc::ld32(tX + lanes, x);
      tc::ld32(tX + lanes + 32, x + 32);
      if (half == 1) {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          x[2 * c] += bf16_lo(qv[c]);
          x[2 * c + 1] += bf16_hi(qv[c]);
        }
      }
      if (g + 1 < ng) {
        uint32_t xb[32];
        if (half == 1) {
#pragma unroll
          for (int c = 0; c < 32; ++c) xb[c] = __float_as_uint(x[c]);
          tc::st32(tX + lanes, xb);
#pragma unroll
          for (int c = 0; c < 32; ++c) xb[c] = __float_as_uint(x[32 + c]);
          tc::st32(tX + lanes + 32, xb);
        }
#pragma unroll
        for (int c = 0; c < 32; ++c) xb[c] = pack_bf16(x[2 * c], x[2 * c + 1]);
        tc::st32(tXb + lanes, xb);
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(xready);
        if (half == 1 && !(ok = convert(g + 1))) break;
      } else {
        // (A_s or B_s)[i][jc] = X^T[r][i]
        float* out = p.seg_maps + (static_cast<size_t>(unit) * maps + seg) * 2 * kD * kD + half * kD * kD;
#pragma unroll
        for (int i = 0; i < 64; ++i) out[i * kD + jc] = x[i];
      }
    }
    if (!ok) {
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
  const int items = p.units * p.seg_num;
  if (items == 0) return cudaSuccess;
  // The attribute belongs to the current device: set it on every launch, as the
  // other large-shared-memory launchers do (a process may drive several GPUs).
  const cudaError_t e =
      cudaFuncSetAttribute(linear_seg_affine_wy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  linear_seg_affine_wy_kernel<<<items, kThreads, kSmemBytes, stream>>>(mk64, mv64, p);
  return cudaGetLastError();
}

}  // namespace ttt
