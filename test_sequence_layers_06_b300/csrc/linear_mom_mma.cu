// TTT-Linear with momentum gradient descent, bf16 inputs, d = 64, b a multiple of
// 16, on the tensor cores: one CTA per (batch row, head), W and the momentum M
// resident in registers across the sequence.
//
// Method (the E²-TTT write-up, "推理时的“临阵磨枪”：Test-Time Training如何教会AI“边做边学”",
// sections 2.3 and 5.1, as the oracle reads it: token-level momentum with the
// gradients taken at the chunk-start weights). For a chunk of n tokens with start
// (W_a, M_a), E = K W_a - V and, after its s-th token,
//   M_s = beta^s M_a + (1 - beta) sum_{i<=s} beta^(s-i) k_i^T e_i,
//   W_s = W_a - alpha [c_s M_a + sum_{i<=s} (1 - beta^(s-i+1)) k_i^T e_i],
//   c_s = beta + ... + beta^s,   z_s = q_s W_s,
// so Z = Q W_a - alpha c .* (Q M_a) - alpha (tril(Q K^T) .* D) E with
// D[s][i] = 1 - beta^(s-i+1), and the chunk's end state is row s = n.
//
// Layout as the TTT-Linear read-out (linear_mma.cu): each of 4 consumer warps owns
// 16 output columns j and keeps W^T and M^T (16 x 64 each) as fp32 mma.sync
// accumulator fragments; everything is written transposed, so that
//   E^T = W_a^T K^T - V^T
//   Z^T = W_a^T Q^T + (-alpha c) .* (M_a^T Q^T) + (-alpha E^T) (S .* D)^T
//   W^T += (-alpha c_n) M_a^T + (-alpha E^T .* d) K,     d_i = 1 - beta^(n-i+1)
//   M^T  = beta^n M_a^T + ((1 - beta) E^T .* w) K,      w_i = beta^(n-i)
// (the column scalings act on the token index of E^T's C fragment before it is
// packed as the A operand). These are the token recurrence solved over any run of
// tokens that share one W_a, so a chunk larger than 16 tokens is walked in 16-token
// tiles: E of every tile from the chunk-start W (a kept bf16 copy), the rest from
// the running (W, M) with the tile's own c, D, d and w (b = 16: every tile is a
// chunk). A producer warp streams the Q, K, V tiles by TMA into
// a 6-stage ring and forms (S .* D)^T once per tile for the consumers. Every wait
// is bounded in wall-clock time. Powers of beta are products in fp32, as a table.
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
constexpr int kZOff = kStages * kStageBytes;
constexpr int kZBytes = kTile * 16 * 2;       // 512 per warp and buffer
constexpr int kSOff = kZOff + kWarps * 2 * kZBytes;  // per stage: (S .* D)^T B fragments, 16 bytes per lane
constexpr int kSBytes = 32 * 16;
constexpr int kPowOff = kSOff + kStages * kSBytes;   // beta^0 .. beta^17, fp32
constexpr int kBarOff = kPowOff + 128;
constexpr int kAbortOff = kBarOff + 3 * kStages * 8;
constexpr int kSmemBytes = kAbortOff + 16 + 1024;    // + slack to align the base to 1024
static_assert(kSmemBytes <= 48 * 1024, "no opt-in to more dynamic shared memory");

enum : int { kWhereMomProducer = 50, kWhereMomConsumer = 51 };

// kTileChunk: every 16-token tile is a whole chunk (b = 16), so the chunk-start copy of W^T is the
// running one and no second copy is kept; otherwise a tile's error uses the chunk-start copy.
template <bool kTileChunk>
__global__ void __launch_bounds__(kThreads, 2)
    linear_mom_mma_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                          const __grid_constant__ CUtensorMap mv, MomParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* empty = full + kStages;
  uint64_t* sready = empty + kStages;  // the tile's (S .* D)^T fragments are written
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kAbortOff);
  float* pw = reinterpret_cast<float*>(smem + kPowOff);

  const int unit = blockIdx.x;
  const int h = unit % p.H;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_tiles = (p.T + kTile - 1) / kTile;
  const float beta = p.beta[h];

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps);
      mbar_init(&sready[s], 1);
    }
    *abort_flag = 0;
    float x = 1.f;
    for (int k = 0; k < 18; ++k) {
      pw[k] = x;
      x *= beta;
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kWarps) {
    // ------------------------------------------------------------ producer
    const int g = lane >> 2, tg = lane & 3, mi = lane >> 3, mr = lane & 7;
    // Decay factors of this lane's elements (t = g (+8), t' = 8nt + 2tg (+1)); zero above the diagonal.
    float dm[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int t = g + 8 * (r >> 1), t2 = 8 * nt + 2 * tg + (r & 1);
        dm[nt][r] = t2 <= t ? 1.f - pw[t - t2 + 1] : 0.f;
      }
    int issued = 0;  // lane 0
    auto load = [&](int u) {
      const int s = u % kStages;
      mbar_arrive_expect_tx(&full[s], kStageBytes);
      uint8_t* st = smem + s * kStageBytes;
      tma_load_3d(st, &mq, &full[s], 0, u * kTile, unit);
      tma_load_3d(st + kTileBytes, &mk, &full[s], 0, u * kTile, unit);
      tma_load_3d(st + 2 * kTileBytes, &mv, &full[s], 0, u * kTile, unit);
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
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) sacc[nt][r] *= dm[nt][r];
      // (S .* D)'s C fragment (rows t, columns t') is the B fragment (k = t', n = t) of its transpose.
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
        if (!*abort_flag) report_error(p.status, TTT_ERR_TIMEOUT, kWhereMomProducer, unit);
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
  const int mi = lane >> 3;
  const int mr = lane & 7;
  const float nalpha = -p.alpha[h];
  __nv_bfloat16* Zg = static_cast<__nv_bfloat16*>(p.Z);

  // Token columns of this lane's C fragments: 8 nt + 2 tg + r2. -alpha c for the read-out.
  float cz[2][2];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int r2 = 0; r2 < 2; ++r2) {
      const int col = 8 * nt + 2 * tg + r2;
      float c = 0.f;
      for (int j = 1; j <= col + 1; ++j) c += pw[j];
      cz[nt][r2] = nalpha * c;
    }
  // End-of-chunk factors for a chunk of n tokens: -alpha d and (1 - beta) w per token column,
  // -alpha c_n and beta^n.
  float dd[2][2], ww[2][2], ncn = 0.f, bn = 1.f;
  auto set_chunk = [&](int n) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int r2 = 0; r2 < 2; ++r2) {
        const int col = 8 * nt + 2 * tg + r2;
        dd[nt][r2] = col < n ? nalpha * (1.f - pw[n - col]) : 0.f;
        ww[nt][r2] = col < n ? (1.f - beta) * pw[n - 1 - col] : 0.f;
      }
    float c = 0.f;
    for (int j = 1; j <= n; ++j) c += pw[j];
    ncn = nalpha * c;
    bn = pw[n];
  };
  set_chunk(kTile);

  // W^T and M^T fragments: [q] covers input columns i in [8q, 8q+8) of rows j = jw+g, jw+g+8.
  float Wt[8][4], Mt[8][4];
  {
    const float* W0 = p.W0 + static_cast<size_t>(h) * kD * kD;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int i = 8 * q + 2 * tg;
      Wt[q][0] = W0[i * kD + jw + g];
      Wt[q][1] = W0[(i + 1) * kD + jw + g];
      Wt[q][2] = W0[i * kD + jw + g + 8];
      Wt[q][3] = W0[(i + 1) * kD + jw + g + 8];
#pragma unroll
      for (int r = 0; r < 4; ++r) Mt[q][r] = 0.f;
    }
  }

  uint32_t wa[4][4];  // bf16 A fragments of the chunk-start W^T (not kept when every tile is a chunk)
  for (int u = 0; u < num_tiles; ++u) {
    const int s = u % kStages;
    if (!mbar_wait_or_abort(&sready[s], (u / kStages) & 1, p.timeout_ns, abort_flag)) {
      if (!*abort_flag) report_error(p.status, TTT_ERR_TIMEOUT, kWhereMomConsumer, unit);
      *abort_flag = 1;
      break;
    }
    const uint4 sv = *reinterpret_cast<const uint4*>(smem + kSOff + s * kSBytes + lane * 16);
    const uint32_t sQ = smem_u32(smem + s * kStageBytes);
    const uint32_t sK = sQ + kTileBytes;
    const uint32_t sV = sQ + 2 * kTileBytes;
    if (u == num_tiles - 1 && p.T - u * kTile < kTile) set_chunk(p.T - u * kTile);  // a ragged last chunk

    // bf16 A fragments of the tile-start (running) W^T and M^T (k-step k: i in [16k, 16k+16)).
    uint32_t wr[4][4], mra[4][4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      wr[k][0] = pack_bf16(Wt[2 * k][0], Wt[2 * k][1]);
      wr[k][1] = pack_bf16(Wt[2 * k][2], Wt[2 * k][3]);
      wr[k][2] = pack_bf16(Wt[2 * k + 1][0], Wt[2 * k + 1][1]);
      wr[k][3] = pack_bf16(Wt[2 * k + 1][2], Wt[2 * k + 1][3]);
      mra[k][0] = pack_bf16(Mt[2 * k][0], Mt[2 * k][1]);
      mra[k][1] = pack_bf16(Mt[2 * k][2], Mt[2 * k][3]);
      mra[k][2] = pack_bf16(Mt[2 * k + 1][0], Mt[2 * k + 1][1]);
      mra[k][3] = pack_bf16(Mt[2 * k + 1][2], Mt[2 * k + 1][3]);
    }
    if constexpr (!kTileChunk) {
      if ((u * kTile) % p.b == 0) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int r = 0; r < 4; ++r) wa[k][r] = wr[k][r];
      }
    }

    // -V^T as the accumulator of E^T (ldmatrix.trans of V's 8x8 blocks gives the C-fragment pairs).
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
    // E^T = W_a^T K^T - V^T (K as the B operand, k = i, n = t), in two partial sums.
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t r[4];
      ldsm_x4(r, sK + swz128(((mi >> 1) << 3) + mr, 2 * k + (mi & 1)));
      const uint32_t b0[2] = {r[0], r[1]}, b1[2] = {r[2], r[3]};
      mma_bf16_16816(k < 2 ? e[0] : e2[0], kTileChunk ? wr[k] : wa[k], b0);
      mma_bf16_16816(k < 2 ? e[1] : e2[1], kTileChunk ? wr[k] : wa[k], b1);
    }
    // K as the B operand of the updates (k = t, n = i): kbt[q] for i in [8q, 8q+8).
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
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) e[nt][r] += e2[nt][r];

    // E^T scaled per token column, as A operands (m = j, k = t): -alpha E^T for the read-out,
    // -alpha E^T .* d for W, (1 - beta) E^T .* w for M.
    uint32_t ea[4], ed[4], em[4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      ea[2 * nt] = pack_bf16(nalpha * e[nt][0], nalpha * e[nt][1]);
      ea[2 * nt + 1] = pack_bf16(nalpha * e[nt][2], nalpha * e[nt][3]);
      ed[2 * nt] = pack_bf16(dd[nt][0] * e[nt][0], dd[nt][1] * e[nt][1]);
      ed[2 * nt + 1] = pack_bf16(dd[nt][0] * e[nt][2], dd[nt][1] * e[nt][3]);
      em[2 * nt] = pack_bf16(ww[nt][0] * e[nt][0], ww[nt][1] * e[nt][1]);
      em[2 * nt + 1] = pack_bf16(ww[nt][0] * e[nt][2], ww[nt][1] * e[nt][3]);
    }

    // The state update first (the chain to the next tile): W^T with the start momentum, then M^T.
#pragma unroll
    for (int q = 0; q < 8; ++q) {
#pragma unroll
      for (int r = 0; r < 4; ++r) Wt[q][r] = fmaf(ncn, Mt[q][r], Wt[q][r]);
      mma_bf16_16816(Wt[q], ed, kbt[q]);
#pragma unroll
      for (int r = 0; r < 4; ++r) Mt[q][r] *= bn;
      mma_bf16_16816(Mt[q], em, kbt[q]);
    }

    // Read-out: Z^T = W_a^T Q^T + (-alpha c) .* (M_a^T Q^T) + (-alpha E^T) (S .* D)^T.
    float z[2][4] = {}, zm[2][4] = {};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t r[4];
      ldsm_x4(r, sQ + swz128(((mi >> 1) << 3) + mr, 2 * k + (mi & 1)));
      const uint32_t qb0[2] = {r[0], r[1]}, qb1[2] = {r[2], r[3]};
      mma_bf16_16816(z[0], wr[k], qb0);
      mma_bf16_16816(z[1], wr[k], qb1);
      mma_bf16_16816(zm[0], mra[k], qb0);
      mma_bf16_16816(zm[1], mra[k], qb1);
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      z[nt][0] = fmaf(cz[nt][0], zm[nt][0], z[nt][0]);
      z[nt][1] = fmaf(cz[nt][1], zm[nt][1], z[nt][1]);
      z[nt][2] = fmaf(cz[nt][0], zm[nt][2], z[nt][2]);
      z[nt][3] = fmaf(cz[nt][1], zm[nt][3], z[nt][3]);
    }
    const uint32_t sb0[2] = {sv.x, sv.y}, sb1[2] = {sv.z, sv.w};
    mma_bf16_16816(z[0], ea, sb0);
    mma_bf16_16816(z[1], ea, sb1);

    // Every register loaded from the stage has been consumed: hand it back to the producer
    // (the proxy fence orders these reads before its next TMA write).
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);

    // Z^T (rows j, columns t) -> Z[t][j] through the warp's staging tile (transposing stmatrix).
    uint8_t* zbuf = smem + kZOff + (warp * 2 + (u & 1)) * kZBytes;
    {
      uint32_t zr[4] = {pack_bf16(z[0][0], z[0][1]), pack_bf16(z[0][2], z[0][3]),
                        pack_bf16(z[1][0], z[1][1]), pack_bf16(z[1][2], z[1][3])};
      stsm_x4_t(smem_u32(zbuf) + (((mi >> 1) << 3) + mr) * 32 + (mi & 1) * 16, zr);
    }
    __syncwarp();
    {
      const int tok = u * kTile + (lane >> 1);
      const uint4 zv = *reinterpret_cast<const uint4*>(zbuf + (lane >> 1) * 32 + (lane & 1) * 16);
      if (tok < p.T)
        *reinterpret_cast<uint4*>(Zg + (static_cast<size_t>(unit) * p.T + tok) * kD + jw + 8 * (lane & 1)) = zv;
    }
  }

  // Final states, W_out[unit][i][j] and M_out[unit][i][j].
  float* Wo = p.W_out + static_cast<size_t>(unit) * kD * kD;
  float* Mo = p.M_out + static_cast<size_t>(unit) * kD * kD;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int i = 8 * q + 2 * tg;
    Wo[i * kD + jw + g] = Wt[q][0];
    Wo[(i + 1) * kD + jw + g] = Wt[q][1];
    Wo[i * kD + jw + g + 8] = Wt[q][2];
    Wo[(i + 1) * kD + jw + g + 8] = Wt[q][3];
    Mo[i * kD + jw + g] = Mt[q][0];
    Mo[(i + 1) * kD + jw + g] = Mt[q][1];
    Mo[i * kD + jw + g + 8] = Mt[q][2];
    Mo[(i + 1) * kD + jw + g + 8] = Mt[q][3];
  }
}

}  // namespace

bool linear_mom_mma_supported(int d, int b, bool bf16) { return bf16 && d == kD && b > 0 && b % kTile == 0; }

int linear_mom_mma_tile_rows() { return kTile; }

cudaError_t launch_linear_mom_mma(const MomParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                                  const CUtensorMap& mv, cudaStream_t stream) {
  if (p.units == 0) return cudaSuccess;
  if (p.b == kTile)
    linear_mom_mma_kernel<true><<<p.units, kThreads, kSmemBytes, stream>>>(mq, mk, mv, p);
  else
    linear_mom_mma_kernel<false><<<p.units, kThreads, kSmemBytes, stream>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace ttt
