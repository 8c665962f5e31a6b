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
// columns in its own shared memory and hands it to the peer's with one 1 KB bulk
// copy, whose bytes complete a transaction count on the peer's mbarrier. So both
// CTAs hold all four quarters of G; Z's blocks go to the CTA that writes those 32
// columns of Z (staged, then copied, when that is the peer).
//
// Neighbouring tiles overlap: tile u + 1's U/A/P/S (and Q W1 of its Hq) need only
// tile u's W1 update, so they run in the phase of tile u's Z partials, and tile u's
// Z sum runs in the phase of tile u + 1's G partials; a tile takes four CTA
// barriers. A, the bf16 W2 copy and the exchange buffers are double-buffered by
// tile parity and every mbarrier wait is bounded. Each exchange barrier's phase is
// armed (expect_tx) after its buffer's last read, and that read precedes, through
// the chain of exchanges, the peer's next send into it. A cluster barrier at the
// start (the peer's barriers are initialised and armed) and at the end (no copy
// still targets an exited CTA) are the only unbounded waits; both CTAs always
// reach both.
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
// shared memory map (bytes from a 1024-aligned base)
constexpr int kQKV = 0;                                  // [2 stages][Q, K, V]
constexpr int kW1b = kQKV + 2 * 3 * kTileBytes;          // W1[:, own], bf16 [64][128]
constexpr int kW2b = kW1b + kD * kRowH;                  // [2 parity] W2[own, :], bf16 [128][64]
constexpr int kW2bBytes = kMh * 128;
constexpr int kAb = kW2b + 2 * kW2bBytes;                // [2 parity] A, bf16 [16][128]
constexpr int kAbBytes = kTile * kRowH;
constexpr int kAqb = kAb + 2 * kAbBytes;                 // Aq, bf16 [16][128]
constexpr int kGb = kAqb + kTile * kRowH;                // G, bf16 [16][64]
constexpr int kSb = kGb + kTile * 128;                   // tril(Q K^T), bf16 [16][16] in 128-byte rows
constexpr int kBlk = kTile * 16;                         // floats of a 16 x 16 fp32 block (1 KB)
constexpr int kBlkS = kBlk + 16;                         // block stride: neighbouring blocks 64 B apart in banks
constexpr int kPartG = kSb + kTile * 128;                // [2 parity][4 quarters][4 column blocks] blocks
constexpr int kPartGBytes = 16 * kBlkS * 4;
constexpr int kPartZ = kPartG + 2 * kPartGBytes;         // [2 parity][4 quarters][2 column blocks] blocks
constexpr int kPartZBytes = 8 * kBlkS * 4;
constexpr int kZStage = kPartZ + 2 * kPartZBytes;        // [2 parity][2 quarters][2 column blocks]: Z for the peer
constexpr int kZStageBytes = 4 * kBlkS * 4;
constexpr int kBar = kZStage + 2 * kZStageBytes;         // full[2], gfull[2], zfull[2]
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
// A shared-memory block of this CTA to the peer's; its arrival completes `bytes` of the
// transaction count of the peer's mbarrier.
__device__ __forceinline__ void bulk_to_peer(uint32_t remote, uint32_t local, uint32_t bytes, uint32_t remote_bar) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   remote),
               "r"(local), "r"(bytes), "r"(remote_bar)
               : "memory");
}
// Float offset of (row r, column c) in a 16 x 16 fp32 block: 16-byte chunks XOR-swizzled by row pair.
__device__ __forceinline__ int blk_off(int r, int c) { return r * 16 + ((((c >> 2) ^ (r >> 1)) & 3) << 2) + (c & 3); }
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
  // bf16 copies of this warp's slices (local hidden index 16 * warp); W2's by tile parity.
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
  auto store_w2 = [&](int par) {
    uint8_t* base = sm + kW2b + par * kW2bBytes;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      *reinterpret_cast<uint32_t*>(base + swz(16 * warp + g, nt, 128) + 4 * tg) = pack_bf16(w2[nt][0], w2[nt][1]);
      *reinterpret_cast<uint32_t*>(base + swz(16 * warp + g + 8, nt, 128) + 4 * tg) =
          pack_bf16(w2[nt][2], w2[nt][3]);
    }
  };
  store_w1();
  store_w2(0);
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
  if (tid == 0 && n_tiles > 0 && p.inject_stall != 1) {  // test hook: the loads never start
    prefetch_tmap(&mq);
    prefetch_tmap(&mk);
    prefetch_tmap(&mv);
    load_tile(0);
    if (n_tiles > 1) load_tile(1);
  }

  const uint32_t W1b = s0 + kW1b, Aqb = s0 + kAqb, Gb = s0 + kGb, Sb = s0 + kSb;
  // The peer's exchange barriers (parity s at + 8 s bytes: the window maps offsets linearly).
  const uint32_t gbar_peer = map_peer(smem_u32(&gfull[0]), peer), zbar_peer = map_peer(smem_u32(&zfull[0]), peer);

  // Tile v's U = K W1, A = gelu(U) (into the A copy of its parity) and P = gelu'(U) (registers)
  // for this warp's hidden units; warps 0 and 1 form one n-tile each of tril(Q K^T).
  float cp[2][4], cq[2][4];
  auto phase_u = [&](int v) {
    const uint32_t sQ = s0 + kQKV + (v & 1) * 3 * kTileBytes, sK = sQ + kTileBytes;
    float cu[2][4] = {};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) cq[nt][r] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      uint32_t a[4], b[4], aq[4];
      ldA(a, sK, 128, 0, 2 * ks, lane);
      ldA(aq, sQ, 128, 0, 2 * ks, lane);
      ldBT(b, W1b, kRowH, 16 * ks, 2 * warp, lane);
      mma2(cu, a, b);
      mma2(cq, aq, b);
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) gelu2(cu[nt][r], cu[nt][r], cp[nt][r]);
    st_tile(sm + kAb + (v & 1) * kAbBytes, kRowH, 0, warp, cu, lane);
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
      *reinterpret_cast<uint32_t*>(sm + kSb + swz(g, nt, 128) + 4 * tg) = pack_bf16(cs[0], cs[1]);
      *reinterpret_cast<uint32_t*>(sm + kSb + swz(g + 8, nt, 128) + 4 * tg) = pack_bf16(cs[2], cs[3]);
    }
  };
  // Tile v's stage has landed (bounded wait).
  auto wait_stage = [&](int v) {
    const bool got = mbar_wait_bounded(&full[v & 1], static_cast<uint32_t>(v >> 1) & 1u, p.timeout_ns);
    if (!got) report_error(p.status, TTT_ERR_TIMEOUT, kWhereClLoad, unit);
    fence_proxy_async_smem();
    return got;
  };
  // Z of tile v for this CTA's 32 columns: the peer's blocks (bounded wait) and ours.
  auto z_sum = [&](int v) {
    const bool got = mbar_wait_bounded(&zfull[v & 1], static_cast<uint32_t>(v >> 1) & 1u, p.timeout_ns);
    if (!got) {
      report_error(p.status, TTT_ERR_TIMEOUT, kWhereClZ, unit);
      return false;
    }
    const float* pz = partZ + (v & 1) * (kPartZBytes / 4);
    const int t = tid >> 4, j = (tid & 15) * 2;
    float2 z = make_float2(0.f, 0.f);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 w = *reinterpret_cast<const float2*>(pz + (q * 2 + (j >> 4)) * kBlkS + blk_off(t, j & 15));
      z.x += w.x;
      z.y += w.y;
    }
    const int tt = v * kTile + t;
    if (tt < p.T) {
      __nv_bfloat16* Z = static_cast<__nv_bfloat16*>(p.Z) + (static_cast<size_t>(unit) * p.T + tt) * kD +
                         32 * static_cast<int>(rank) + j;
      *reinterpret_cast<uint32_t*>(Z) = pack_bf16(z.x, z.y);
    }
    return true;
  };

  // Neighbouring tiles overlap: tile u + 1's U/A/P/S (which needs only the W1 update of tile u)
  // runs in the phase of tile u's Z partials, and tile u's Z sum in the phase of tile u + 1's
  // G partials, so a tile takes four CTA barriers and neither exchange waits on its own phase.
  bool ok = n_tiles > 0;
  if (ok) {
    const bool got = wait_stage(0);
    if (__syncthreads_or(!got)) ok = false;
    else phase_u(0);
  }
  bool stage_ok = true;
  for (int u = 0; ok && u < n_tiles; ++u) {
    const int s = u & 1;
    const uint32_t ph = static_cast<uint32_t>(u >> 1) & 1u;
    const uint32_t sQ = s0 + kQKV + s * 3 * kTileBytes, sK = sQ + kTileBytes;
    const uint8_t* sVp = sm + kQKV + s * 3 * kTileBytes + 2 * kTileBytes;
    const uint32_t Ab = s0 + kAb + s * kAbBytes, W2b = s0 + kW2b + s * kW2bBytes;
    float* pg = partG + s * (kPartGBytes / 4);
    float* pz = partZ + s * (kPartZBytes / 4);

    // A, P and S of tile u are complete, the W2 copy of parity s holds tile u's start weights,
    // and this CTA's Z blocks of tile u - 1 are written.
    if (__syncthreads_or(!stage_ok)) {
      ok = false;
      break;
    }

    // (1) This CTA's quarter kq = w >> 2 of G for value columns [16 np, +16), np = w & 3,
    //     into quarter slot 2 rank + kq of both CTAs; then tile u - 1's Z.
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
      float* blk = pg + ((2 * static_cast<int>(rank) + kq) * 4 + np) * kBlkS;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int c = 8 * nt + 2 * tg;
        *reinterpret_cast<float2*>(blk + blk_off(g, c)) = make_float2(cg[nt][0], cg[nt][1]);
        *reinterpret_cast<float2*>(blk + blk_off(g + 8, c)) = make_float2(cg[nt][2], cg[nt][3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      // (Test hook 2: the second CTA withholds its G blocks, so the first CTA's exchange wait runs out.)
      if (lane == 0 && !(p.inject_stall == 2 && rank == 1))
        bulk_to_peer(map_peer(smem_u32(blk), peer), smem_u32(blk), kBlk * 4, gbar_peer + 8u * s);
    }
    const bool zok = u == 0 || z_sum(u - 1);
    // The peer's two quarters of G (bounded wait) and this CTA's (the barrier).
    const bool gok = mbar_wait_bounded(&gfull[s], ph, p.timeout_ns);
    if (!gok) report_error(p.status, TTT_ERR_TIMEOUT, kWhereClG, unit);
    if (__syncthreads_or(!gok || !zok)) {
      ok = false;
      break;
    }
    // The Z blocks of tile u - 1 are read: arm their slots for tile u + 1.
    if (tid == 0 && u >= 1 && u + 1 < n_tiles) mbar_arrive_expect_tx(&zfull[s ^ 1], kZRecv);

    // (2) G = the sum of the four quarters - V, bf16 (four columns per thread).
    {
      const int t = tid >> 4, j = (tid & 15) * 4;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 v = *reinterpret_cast<const float4*>(pg + (q * 4 + (j >> 4)) * kBlkS + blk_off(t, j & 15));
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

    // (3) D = (G W2^T) .* P and the W2 update; Hq, Aq and the W1 update (this warp's hidden units).
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
      float cs[2][4] = {};
      {
        uint32_t a[4];
        ldA(a, Sb, 128, 0, 0, lane);
        mma2(cs, a, bd);
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) cq[nt][r] = gelu1(fmaf(-eta, cs[nt][r], cq[nt][r]));
      st_tile(sm + kAqb, kRowH, 0, warp, cq, lane);
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
    __syncthreads();  // Aq complete; the stage of tile u is read
    if (tid == 0 && u + 2 < n_tiles) load_tile(u + 2);

    // (4) Quarter kq's block of Z for value columns [16 np, +16) (with its block of
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
      // Its slot in the owner's Z blocks; a block for the peer is staged here first.
      float* slot = pz + ((2 * static_cast<int>(rank) + kq) * 2 + (np & 1)) * kBlkS;
      const bool local = static_cast<uint32_t>(np >> 1) == rank;
      float* blk = local ? slot : reinterpret_cast<float*>(sm + kZStage + s * kZStageBytes) + (kq * 2 + (np & 1)) * kBlkS;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int c = 8 * nt + 2 * tg;
        *reinterpret_cast<float2*>(blk + blk_off(g, c)) = make_float2(cz[nt][0], cz[nt][1]);
        *reinterpret_cast<float2*>(blk + blk_off(g + 8, c)) = make_float2(cz[nt][2], cz[nt][3]);
      }
      if (!local) {
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) bulk_to_peer(map_peer(smem_u32(slot), peer), smem_u32(blk), kBlk * 4, zbar_peer + 8u * s);
      }
    }
    // Tile u + 1's U/A/P/S, and this warp's rows of the updated W2 into the copy of parity s ^ 1
    // (its last reads, tile u - 1's, preceded this tile's first barrier).
    if (u + 1 < n_tiles) {
      stage_ok = wait_stage(u + 1);
      if (stage_ok) phase_u(u + 1);
    }
    store_w2(s ^ 1);
  }
  // The last tile's Z: this CTA's blocks are written (the barrier), the peer's are awaited.
  __syncthreads();
  if (ok && !z_sum(n_tiles - 1)) ok = false;
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
