// C ABI of the chunked TTT scan: argument checks, workspace layout, TMA
// descriptors and kernel dispatch. Declarations and contracts: include/ttt.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <algorithm>
#include <cstring>
#include <initializer_list>
#include <mutex>

#include "ttt.h"
#include "kernels.h"
#include "ttt_device.cuh"

namespace {

using ttt::kStatusBytes;

constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;  // 2 s
constexpr int kMaxD = 64;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool sizes_ok(int B, int H, int T, int d, int b) {
  if (B < 1 || H < 1 || T < 0 || d < 1 || b < 1) return false;
  // Every flat index of [B][H][T][d] must fit a signed 64-bit offset and every
  // TMA coordinate a signed 32-bit one.
  const long double n = static_cast<long double>(B) * H * T * d;
  return n < 9.0e18L && static_cast<long double>(B) * H < 2147483647.0L;
}

size_t mlp_hidden(int d) { return static_cast<size_t>(4) * d; }

// A buffer the call touches: start and length in bytes.
struct Span {
  const void* p;
  size_t n;
};

bool overlap(const Span& a, const Span& b) {
  if (a.p == nullptr || b.p == nullptr || a.n == 0 || b.n == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
  return a0 < b0 + b.n && b0 < a0 + a.n;
}

// Outputs (and scratch) may overlap neither an input nor one another; inputs
// may alias each other, since they are only read.
bool outputs_disjoint(std::initializer_list<Span> outs, std::initializer_list<Span> ins) {
  for (auto o = outs.begin(); o != outs.end(); ++o) {
    for (const Span& i : ins)
      if (overlap(*o, i)) return false;
    for (auto o2 = o + 1; o2 != outs.end(); ++o2)
      if (overlap(*o, *o2)) return false;
  }
  return true;
}

// Bytes of a [n0][n1][n2][n3] tensor with elements of `es` bytes.
size_t bytes4(int n0, int n1, int n2, int n3, size_t es) {
  return static_cast<size_t>(n0) * n1 * n2 * n3 * es;
}

ttt_options defaults(const ttt_options* opt) {
  ttt_options o;
  std::memset(&o, 0, sizeof(o));
  if (opt) o = *opt;
  if (o.wait_timeout_ns == 0) o.wait_timeout_ns = kDefaultTimeoutNs;
  return o;
}

// Streaming multiprocessors of the current device (148 on a B300 if the query fails).
int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

// How TTT-Linear runs: which kernel, and for the segment-parallel form how the
// sequence is cut. A plan with seg_count == 1 is one pass over every sequence.
struct LinearPlan {
  bool mma;       // tensor-core kernels (bf16, d = 64, b % 16 == 0); else fp32 SIMT
  int seg_len;    // tokens per segment (a multiple of b)
  int seg_count;  // segments per (batch row, head)
  bool affine_wy; // affine maps on tcgen05 in 64-token steps (else warp-level MMAs)
  int pieces;     // segment pieces: the affine maps of piece p + 1 overlap the read-out of piece p
};

constexpr int kSegMinTokens = 256;  // shortest segment the automatic plan makes
constexpr int kMmaCtasPerSm = 3;    // linear_mma_kernel's occupancy (its launch bounds)
constexpr int kAutoPieces = 1;      // pieces of the automatic plan

ttt_status plan_linear(int B, int H, int T, int d, int b, bool bf16, const ttt_options& o, LinearPlan* out) {
  LinearPlan pl{false, T > 0 ? T : 1, 1, false, 1};
  if (o.pieces < 0) return TTT_ERR_ARG;
  const bool mma_ok = d == 64 && b % 16 == 0 && bf16;
  if (o.force_path == 2 && !mma_ok) return TTT_ERR_UNSUPPORTED;
  if (o.force_path == 3 && !mma_ok) return TTT_ERR_UNSUPPORTED;
  if (o.seg_len < 0) return TTT_ERR_ARG;
  if (o.seg_len > 0 && (o.seg_len % b != 0 || o.seg_len % 16 != 0)) return TTT_ERR_ARG;
  pl.mma = mma_ok && o.force_path != 1 && T > 0;
  if (!pl.mma) {
    *out = pl;
    return TTT_OK;
  }
  const int units = B * H;
  const int slots = kMmaCtasPerSm * sm_count();  // resident read-out CTAs
  bool seg = false;
  if (o.force_path == 3) seg = true;
  if (o.force_path == 0 && units < slots && T >= 2 * kSegMinTokens) seg = true;
  if (seg) {
    long long len = o.seg_len;
    if (len == 0) {
      // Segments hold whole chunks; where the 64-token tensor-core affine kernel
      // applies (b = 16, 32 or a multiple of 64) they also hold whole 64-token steps.
      const long long align = (b % 64 == 0 || 64 % b == 0) ? std::max(b, 64) : b;
      const long long min_len = ((kSegMinTokens + align - 1) / align) * align;
      // The segment count that minimises an estimate of the step: waves of affine-map CTAs
      // (two per SM) and of read-out CTAs (three per SM), each wave as long as one segment
      // at the per-token time one CTA of that kernel measured at full occupancy, plus the
      // combine's chain over the segment boundaries. Partial waves count as whole ones.
      const double aff_ns = b <= 32 ? 25.0 : (b < 256 ? 19.0 : 12.5), out_ns = 47.0, step_ns = 1400.0;
      const long long slots_a = 2LL * sm_count(), slots_r = slots;
      double best = -1.0;
      for (long long S = 2; S <= T / min_len; ++S) {
        long long L = ((T + S - 1) / S + align - 1) / align * align;
        if (L < min_len) L = min_len;
        const long long cnt = (T + L - 1) / L;
        if (cnt < 2) continue;
        const double waves_a = static_cast<double>((units * (cnt - 1) + slots_a - 1) / slots_a);
        const double waves_r = static_cast<double>((units * cnt + slots_r - 1) / slots_r);
        const double cost = waves_a * L * aff_ns + (cnt - 1) * step_ns + waves_r * L * out_ns;
        if (best < 0.0 || cost < best) {
          best = cost;
          len = L;
        }
      }
      if (len == 0) len = min_len;
    }
    const long long count = (T + len - 1) / len;
    // Grids of one read-out CTA per (unit, segment) and 8 combine CTAs per unit
    // must fit a 32-bit signed count.
    if (static_cast<long long>(units) * std::max(count, 8LL) > 2147483647LL) return TTT_ERR_UNSUPPORTED;
    if (count >= 2) {
      pl.seg_len = static_cast<int>(len);
      pl.seg_count = static_cast<int>(count);
      pl.affine_wy = ttt::linear_seg_wy_supported(b, pl.seg_len);
      // Phase events time each kernel over all segments, so they ask for one piece.
      const int want = o.phase_events ? 1 : (o.pieces > 0 ? o.pieces : kAutoPieces);
      pl.pieces = std::max(1, std::min(want, pl.seg_count));
    }
  }
  *out = pl;
  return TTT_OK;
}

// Bytes of segment scratch: affine maps (A_s, B_s) and start states, both for
// every segment but one, fp32.
size_t seg_scratch_bytes(const LinearPlan& pl, int units, int d) {
  if (pl.seg_count < 2) return 0;
  const size_t per = static_cast<size_t>(units) * (pl.seg_count - 1) * d * d * sizeof(float);
  return 3 * per;
}

// Workspace: [status block 256 B][variant scratch].
size_t workspace_bytes_impl(int B, int H, int T, int d, int b, int variant, const ttt_options* opt) {
  if (!sizes_ok(B, H, T, d, b)) return 0;
  size_t bytes = kStatusBytes;
  if (variant == TTT_VARIANT_MLP) {
    bytes += round_up(ttt::mlp_simt_snapshot_bytes(B * H, d, static_cast<int>(mlp_hidden(d))), 256);
  } else if (variant == TTT_VARIANT_LINEAR) {
    // Sized for bf16 operands, the only dtype whose plan may use segments.
    LinearPlan pl;
    if (plan_linear(B, H, T, d, b, true, defaults(opt), &pl) == TTT_OK) bytes += seg_scratch_bytes(pl, B * H, d);
  } else {
    return 0;
  }
  return bytes;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 3-D map over a [units][T][d] bf16 tensor, box [1][box_t][box_d].
bool encode_3d(CUtensorMap* map, const void* base, int units, int T, int d, int box_t, int box_d,
               CUtensorMapSwizzle swz) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(T > 0 ? T : 1),
                              static_cast<cuuint64_t>(units)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                                 static_cast<cuuint64_t>(T > 0 ? T : 1) * d * 2};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(box_d), static_cast<cuuint32_t>(box_t), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                         box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}


// A second stream per device for the overlapped segment pieces (created once,
// non-blocking; work on it is ordered against the caller's stream by events).
cudaStream_t side_stream() {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static cudaStream_t streams[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (streams[dev] == nullptr && cudaStreamCreateWithFlags(&streams[dev], cudaStreamNonBlocking) != cudaSuccess)
    streams[dev] = nullptr;
  return streams[dev];
}

// The segment-parallel form in `pieces` pieces. Read-out piece p covers segments
// [r_p, r_{p+1}); it needs the start states up to segment r_{p+1} - 1, i.e. the
// maps [0, r_{p+1} - 1). Map piece p covers [max(r_p - 1, 0), r_{p+1} - 1) and its
// combine continues the chain from the start state the previous piece wrote.
//   stream s:    maps 0, combine 0, read-out 0, wait(combine 1), read-out 1, ...
//   side stream: wait(maps 0), maps 1, wait(combine 0), combine 1, maps 2, combine 2, ...
// so the affine maps of piece p + 1 run beside the read-out of piece p. Every
// kernel waits only for work enqueued before it (stream order and events); no
// kernel waits for another that runs at the same time.
template <class MapsFn, class CombineFn, class ReadFn>
cudaError_t run_in_pieces(int S, int pieces, cudaStream_t s, MapsFn maps, CombineFn combine, ReadFn readout) {
  constexpr int kMaxPieces = 64;
  pieces = std::min(pieces, kMaxPieces);
  cudaStream_t x = side_stream();
  if (x == nullptr) return cudaErrorUnknown;
  auto bound = [&](int p) { return static_cast<int>((static_cast<long long>(S) * p) / pieces); };
  // done[p]: the start states of piece p are written; done[pieces]: maps of piece 0 done.
  cudaEvent_t done[kMaxPieces + 1] = {};
  cudaError_t err = cudaSuccess;
  int made = 0;
  for (; made <= pieces && err == cudaSuccess; ++made)
    err = cudaEventCreateWithFlags(&done[made], cudaEventDisableTiming);
  if (err == cudaSuccess) {
    const int m1 = bound(1) - 1;
    if (m1 > 0) err = maps(0, m1, s);
    if (err == cudaSuccess) err = cudaEventRecord(done[pieces], s);
    if (err == cudaSuccess && m1 > 0) err = combine(0, m1, s);
    if (err == cudaSuccess) err = cudaEventRecord(done[0], s);
    if (err == cudaSuccess) err = cudaStreamWaitEvent(x, done[pieces], 0);
    for (int p = 1; p < pieces && err == cudaSuccess; ++p) {
      const int m0 = bound(p) - 1, m1p = bound(p + 1) - 1;
      if (m1p > m0) err = maps(m0, m1p, x);
      if (err == cudaSuccess) err = cudaStreamWaitEvent(x, done[p - 1], 0);
      if (err == cudaSuccess && m1p > m0) err = combine(m0, m1p, x);
      if (err == cudaSuccess) err = cudaEventRecord(done[p], x);
    }
    for (int p = 0; p < pieces && err == cudaSuccess; ++p) {
      if (p > 0) err = cudaStreamWaitEvent(s, done[p], 0);
      if (err == cudaSuccess) err = readout(bound(p), bound(p + 1), s);
    }
  }
  for (int i = 0; i < made; ++i) cudaEventDestroy(done[i]);  // released once their work completes
  return err;
}

ttt_status reset_status(void* ws, cudaStream_t s) {
  return cudaMemsetAsync(ws, 0, sizeof(ttt::StatusBlock), s) == cudaSuccess ? TTT_OK : TTT_ERR_CUDA;
}

}  // namespace

namespace ttt {

// Whether the tensor-core TTT-MLP kernel serves a call with these arguments.
bool mlp_uses_mma(int T, int d, int b, ttt_dtype dt, const ttt_options* opt) {
  MlpParams p;
  std::memset(&p, 0, sizeof(p));
  p.bf16 = dt == TTT_BF16;
  p.d = d;
  p.m = static_cast<int>(mlp_hidden(d));
  p.b = b;
  return mlp_mma_supported(p) && T > 0 && (opt == nullptr || opt->force_path != 1);
}

size_t mlp_workspace_bytes_for_path(int B, int H, int T, int d, int b, ttt_dtype dt, const ttt_options* opt) {
  if (!sizes_ok(B, H, T, d, b)) return 0;
  if (mlp_uses_mma(T, d, b, dt, opt)) return kStatusBytes;  // chunk-start copies stay on chip
  return workspace_bytes_impl(B, H, T, d, b, TTT_VARIANT_MLP, nullptr);
}

// Checks, workspace layout and launch of a TTT-MLP forward. With ws_by_path the
// workspace need only cover the kernel that serves the call; otherwise it must
// cover ttt_workspace_bytes() (every kernel).
ttt_status mlp_forward(const void* Q, const void* K, const void* V, ttt_dtype dt, const float* eta,
                       const float* W1_0, const float* W2_0, int B, int H, int T, int d, int b, void* Z,
                       float* W1_out, float* W2_out, void* workspace, size_t ws_bytes, void* stream,
                       const ttt_options* opt, bool ws_by_path) {
  if (dt != TTT_F32 && dt != TTT_BF16) return TTT_ERR_ARG;
  if (!sizes_ok(B, H, T, d, b)) return TTT_ERR_ARG;
  if (d > kMaxD) return TTT_ERR_UNSUPPORTED;
  if (!eta || !W1_0 || !W2_0 || !W1_out || !W2_out || !workspace) return TTT_ERR_ARG;
  if (T > 0 && (!Q || !K || !V || !Z)) return TTT_ERR_ARG;
  for (const void* p : {static_cast<const void*>(Q), static_cast<const void*>(K), static_cast<const void*>(V),
                        static_cast<const void*>(Z), static_cast<const void*>(eta), static_cast<const void*>(W1_0),
                        static_cast<const void*>(W2_0), static_cast<const void*>(W1_out),
                        static_cast<const void*>(W2_out), static_cast<const void*>(workspace)})
    if (p && !aligned16(p)) return TTT_ERR_ARG;
  const ttt_options o = defaults(opt);
  if (o.force_path < 0 || o.force_path > 3) return TTT_ERR_ARG;
  const size_t need = ws_by_path ? mlp_workspace_bytes_for_path(B, H, T, d, b, dt, opt)
                                 : workspace_bytes_impl(B, H, T, d, b, TTT_VARIANT_MLP, nullptr);
  if (need == 0 || ws_bytes < need) return TTT_ERR_ARG;
  {
    const size_t seq = bytes4(B, H, T, d, dt == TTT_BF16 ? 2 : 4);
    const size_t w1 = bytes4(d, static_cast<int>(mlp_hidden(d)), 1, 1, 4);
    if (!outputs_disjoint({{Z, seq}, {W1_out, w1 * B * H}, {W2_out, w1 * B * H}, {workspace, ws_bytes}},
                          {{Q, seq}, {K, seq}, {V, seq}, {eta, bytes4(H, 1, 1, 1, 4)}, {W1_0, w1 * H}, {W2_0, w1 * H}}))
      return TTT_ERR_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  ttt::MlpParams p;
  p.Q = Q; p.K = K; p.V = V; p.Z = Z;
  p.eta = eta; p.W1_0 = W1_0; p.W2_0 = W2_0; p.W1_out = W1_out; p.W2_out = W2_out;
  p.snap = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + kStatusBytes);
  p.B = B; p.H = H; p.T = T; p.d = d; p.m = static_cast<int>(mlp_hidden(d)); p.b = b;
  p.units = B * H;
  p.bf16 = (dt == TTT_BF16);
  p.status = static_cast<ttt::StatusBlock*>(workspace);
  p.timeout_ns = o.wait_timeout_ns;
  p.inject_stall = o.inject_stall;

  const bool mma_ok = ttt::mlp_mma_supported(p);
  const bool cluster_ok = ttt::mlp_cluster_supported(p);
  if (o.force_path == 2 && !mma_ok) return TTT_ERR_UNSUPPORTED;
  if (o.force_path == 3 && !cluster_ok) return TTT_ERR_UNSUPPORTED;
  const bool use_mma = mma_ok && o.force_path != 1 && T > 0;
  // b = 16: two CTAs per unit (a cluster sharing the hidden units) unless one CTA is forced.
  const bool use_cluster = use_mma && cluster_ok && o.force_path != 2;

  ttt_status st = reset_status(workspace, s);
  if (st != TTT_OK) return st;
  cudaError_t err;
  if (use_mma) {
    CUtensorMap mq, mk, mv;
    const int rows = ttt::mlp_mma_tile_rows();
    if (!encode_3d(&mq, Q, p.units, T, d, rows, d, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_3d(&mk, K, p.units, T, d, rows, d, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_3d(&mv, V, p.units, T, d, rows, d, CU_TENSOR_MAP_SWIZZLE_128B))
      return TTT_ERR_CUDA;
    err = use_cluster ? ttt::launch_mlp_cluster(p, mq, mk, mv, s) : ttt::launch_mlp_mma(p, mq, mk, mv, s);
  } else {
    err = ttt::launch_mlp_simt(p, s);
  }
  return err == cudaSuccess ? TTT_OK : TTT_ERR_CUDA;
}


}  // namespace ttt

extern "C" {

size_t ttt_workspace_bytes(int B, int H, int T, int d, int b, int variant) {
  return workspace_bytes_impl(B, H, T, d, b, variant, nullptr);
}

size_t ttt_workspace_bytes_ex(int B, int H, int T, int d, int b, int variant, const ttt_options* opt) {
  return workspace_bytes_impl(B, H, T, d, b, variant, opt);
}

const char* ttt_status_str(ttt_status s) {
  switch (s) {
    case TTT_OK: return "ok";
    case TTT_ERR_ARG: return "invalid argument";
    case TTT_ERR_UNSUPPORTED: return "unsupported request";
    case TTT_ERR_CUDA: return "CUDA runtime error";
    case TTT_ERR_TIMEOUT: return "a kernel wait ran out of time";
    case TTT_ERR_DEVICE_CHECK: return "a kernel consistency check failed";
  }
  return "unknown status";
}

ttt_status ttt_linear_plan(int B, int H, int T, int d, int b, ttt_dtype dt, const ttt_options* opt,
                           ttt_plan* out) {
  if (out == nullptr) return TTT_ERR_ARG;
  if (dt != TTT_F32 && dt != TTT_BF16) return TTT_ERR_ARG;
  if (!sizes_ok(B, H, T, d, b)) return TTT_ERR_ARG;
  if (d > kMaxD) return TTT_ERR_UNSUPPORTED;
  const ttt_options o = defaults(opt);
  if (o.force_path < 0 || o.force_path > 3) return TTT_ERR_ARG;
  LinearPlan pl;
  const ttt_status st = plan_linear(B, H, T, d, b, dt == TTT_BF16, o, &pl);
  if (st != TTT_OK) return st;
  out->path = !pl.mma ? 1 : (pl.seg_count > 1 ? 3 : 2);
  out->seg_len = pl.seg_len;
  out->seg_count = pl.seg_count;
  out->kernels = T == 0 ? 0 : (pl.seg_count > 1 ? 3 : 1);
  out->affine = pl.seg_count > 1 ? (pl.affine_wy ? 2 : 1) : 0;
  out->pieces = pl.pieces;
  if (pl.seg_count > 1) out->kernels = 3 * pl.pieces;
  return TTT_OK;
}

ttt_status ttt_linear_fwd_ex(const void* Q, const void* K, const void* V, ttt_dtype dt, const float* eta,
                             const float* W0, int B, int H, int T, int d, int b, void* Z, float* W_out,
                             void* workspace, size_t ws_bytes, void* stream, const ttt_options* opt) {
  if (dt != TTT_F32 && dt != TTT_BF16) return TTT_ERR_ARG;
  if (!sizes_ok(B, H, T, d, b)) return TTT_ERR_ARG;
  if (d > kMaxD) return TTT_ERR_UNSUPPORTED;
  if (!eta || !W0 || !W_out || !workspace) return TTT_ERR_ARG;
  if (T > 0 && (!Q || !K || !V || !Z)) return TTT_ERR_ARG;
  for (const void* p : {static_cast<const void*>(Q), static_cast<const void*>(K), static_cast<const void*>(V),
                        static_cast<const void*>(Z), static_cast<const void*>(eta), static_cast<const void*>(W0),
                        static_cast<const void*>(W_out), static_cast<const void*>(workspace)})
    if (p && !aligned16(p)) return TTT_ERR_ARG;
  const ttt_options o = defaults(opt);
  if (o.force_path < 0 || o.force_path > 3) return TTT_ERR_ARG;
  LinearPlan pl;
  const ttt_status pst = plan_linear(B, H, T, d, b, dt == TTT_BF16, o, &pl);
  if (pst != TTT_OK) return pst;
  if (ws_bytes < kStatusBytes + seg_scratch_bytes(pl, B * H, d)) return TTT_ERR_ARG;
  {
    const size_t seq = bytes4(B, H, T, d, dt == TTT_BF16 ? 2 : 4);
    if (!outputs_disjoint({{Z, seq}, {W_out, bytes4(B, H, d, d, 4)}, {workspace, ws_bytes}},
                          {{Q, seq}, {K, seq}, {V, seq}, {eta, bytes4(H, 1, 1, 1, 4)}, {W0, bytes4(H, d, d, 1, 4)}}))
      return TTT_ERR_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  ttt::LinearParams p;
  p.Q = Q; p.K = K; p.V = V; p.Z = Z;
  p.eta = eta; p.W0 = W0; p.W_out = W_out;
  p.B = B; p.H = H; p.T = T; p.d = d; p.b = b;
  p.units = B * H;
  p.bf16 = (dt == TTT_BF16);
  p.status = static_cast<ttt::StatusBlock*>(workspace);
  p.timeout_ns = o.wait_timeout_ns;
  p.inject_stall = o.inject_stall;
  p.seg_len = pl.seg_len;
  p.seg_count = pl.seg_count;
  p.seg_maps = nullptr;
  p.seg_starts = nullptr;
  p.affine_wy = pl.affine_wy ? 1 : 0;
  p.seg_first = 0;
  p.seg_num = pl.seg_count;
  if (pl.seg_count > 1) {
    const size_t per = static_cast<size_t>(p.units) * (pl.seg_count - 1) * d * d;
    p.seg_maps = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + kStatusBytes);
    p.seg_starts = p.seg_maps + 2 * per;
  }

  ttt_status st = reset_status(workspace, s);
  if (st != TTT_OK) return st;
  cudaError_t err;
  if (pl.mma) {
    CUtensorMap mq, mk, mv;
    const int rows = ttt::linear_mma_tile_rows();
    if (!encode_3d(&mq, Q, p.units, T, d, rows, d, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_3d(&mk, K, p.units, T, d, rows, d, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_3d(&mv, V, p.units, T, d, rows, d, CU_TENSOR_MAP_SWIZZLE_128B))
      return TTT_ERR_CUDA;
    cudaEvent_t* ev = static_cast<cudaEvent_t*>(o.phase_events);
    CUtensorMap mk64, mv64;
    if (pl.seg_count > 1 && pl.affine_wy) {
      const int rows64 = ttt::linear_seg_wy_rows();
      if (!encode_3d(&mk64, K, p.units, T, d, rows64, d, CU_TENSOR_MAP_SWIZZLE_128B) ||
          !encode_3d(&mv64, V, p.units, T, d, rows64, d, CU_TENSOR_MAP_SWIZZLE_128B))
        return TTT_ERR_CUDA;
    }
    // Affine maps [m0, m1), and their combine, on stream `st`.
    auto maps = [&](int m0, int m1, cudaStream_t st) -> cudaError_t {
      ttt::LinearParams q = p;
      q.seg_first = m0;
      q.seg_num = m1 - m0;
      return pl.affine_wy ? ttt::launch_linear_seg_affine_wy(q, mk64, mv64, st)
                          : ttt::launch_linear_seg_affine(q, mk, mv, st);
    };
    auto combine = [&](int m0, int m1, cudaStream_t st) -> cudaError_t {
      ttt::LinearParams q = p;
      q.seg_first = m0;
      q.seg_num = m1 - m0;
      return ttt::launch_linear_seg_combine(q, st);
    };
    auto readout = [&](int s0, int s1, cudaStream_t st) -> cudaError_t {
      ttt::LinearParams q = p;
      q.seg_first = s0;
      q.seg_num = s1 - s0;
      return ttt::launch_linear_mma(q, mq, mk, mv, st);
    };
    err = ev ? cudaEventRecord(ev[0], s) : cudaSuccess;
    if (err == cudaSuccess && pl.seg_count > 1 && pl.pieces > 1) {
      err = run_in_pieces(pl.seg_count, pl.pieces, s, maps, combine, readout);
    } else {
      const int m = pl.seg_count - 1;
      if (err == cudaSuccess && m > 0) err = maps(0, m, s);
      if (err == cudaSuccess && ev) err = cudaEventRecord(ev[1], s);
      if (err == cudaSuccess && m > 0) err = combine(0, m, s);
      if (err == cudaSuccess && ev) err = cudaEventRecord(ev[2], s);
      if (err == cudaSuccess) err = readout(0, pl.seg_count, s);
    }
    if (err == cudaSuccess && ev) err = cudaEventRecord(ev[3], s);
  } else {
    err = ttt::launch_linear_simt(p, s);
  }
  return err == cudaSuccess ? TTT_OK : TTT_ERR_CUDA;
}

ttt_status ttt_linear_fwd(const void* Q, const void* K, const void* V, ttt_dtype dt, const float* eta,
                          const float* W0, int B, int H, int T, int d, int b, void* Z, float* W_out,
                          void* workspace, size_t ws_bytes, void* stream) {
  return ttt_linear_fwd_ex(Q, K, V, dt, eta, W0, B, H, T, d, b, Z, W_out, workspace, ws_bytes, stream,
                           nullptr);
}

ttt_status ttt_mlp_fwd_ex(const void* Q, const void* K, const void* V, ttt_dtype dt, const float* eta,
                          const float* W1_0, const float* W2_0, int B, int H, int T, int d, int b, void* Z,
                          float* W1_out, float* W2_out, void* workspace, size_t ws_bytes, void* stream,
                          const ttt_options* opt) {
  return ttt::mlp_forward(Q, K, V, dt, eta, W1_0, W2_0, B, H, T, d, b, Z, W1_out, W2_out, workspace, ws_bytes,
                          stream, opt, false);
}

ttt_status ttt_mlp_fwd(const void* Q, const void* K, const void* V, ttt_dtype dt, const float* eta,
                       const float* W1_0, const float* W2_0, int B, int H, int T, int d, int b, void* Z,
                       float* W1_out, float* W2_out, void* workspace, size_t ws_bytes, void* stream) {
  return ttt_mlp_fwd_ex(Q, K, V, dt, eta, W1_0, W2_0, B, H, T, d, b, Z, W1_out, W2_out, workspace, ws_bytes,
                        stream, nullptr);
}

ttt_status ttt_linear_decode(const void* q, const void* k, const void* v, ttt_dtype dt, const float* eta,
                             float* W_anchor, float* W_run, int B, int H, int N, int d, int pos, int b, void* z,
                             void* stream) {
  if (dt != TTT_F32 && dt != TTT_BF16) return TTT_ERR_ARG;
  if (B < 1 || H < 1 || N < 0 || d < 1 || b < 1 || pos < 0) return TTT_ERR_ARG;
  if (static_cast<long double>(B) * H * N * d >= 9.0e18L || static_cast<long long>(B) * H * 4 >= 2147483647LL)
    return TTT_ERR_ARG;
  if (d > kMaxD) return TTT_ERR_UNSUPPORTED;
  if (!eta || !W_anchor || !W_run || (N > 0 && (!q || !k || !v || !z))) return TTT_ERR_ARG;
  for (const void* p : {q, k, v, static_cast<const void*>(z), static_cast<const void*>(eta),
                        static_cast<const void*>(W_anchor), static_cast<const void*>(W_run)})
    if (p && !aligned16(p)) return TTT_ERR_ARG;
  {
    const size_t tok = bytes4(B, H, N, d, dt == TTT_BF16 ? 2 : 4), st = bytes4(B, H, d, d, 4);
    if (!outputs_disjoint({{z, tok}, {W_anchor, st}, {W_run, st}},
                          {{q, tok}, {k, tok}, {v, tok}, {eta, bytes4(H, 1, 1, 1, 4)}}))
      return TTT_ERR_ARG;
  }
  ttt::DecodeParams p;
  p.q = q; p.k = k; p.v = v; p.z = z; p.eta = eta;
  p.W_anchor = W_anchor; p.W_run = W_run;
  p.B = B; p.H = H; p.d = d; p.pos = pos; p.b = b;
  p.N = N;
  p.units = B * H;
  p.bf16 = (dt == TTT_BF16);
  return ttt::launch_linear_decode(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? TTT_OK : TTT_ERR_CUDA;
}

ttt_status ttt_linear_decode_step(const void* q, const void* k, const void* v, ttt_dtype dt, const float* eta,
                                  float* W_anchor, float* W_run, int B, int H, int d, int pos, int b, void* z,
                                  void* stream) {
  if (!q || !k || !v || !z) return TTT_ERR_ARG;
  return ttt_linear_decode(q, k, v, dt, eta, W_anchor, W_run, B, H, 1, d, pos, b, z, stream);
}

// Shared checks and launch of the inner-model variants (linear_variants.cu).
static ttt_status variant_check(int variant, const void* Q, const void* K, const void* V, ttt_dtype dt,
                                const float* rate, const float* mbeta, const float* tok_rate, const float* W0,
                                const float* vec0, const float* vec1, int B, int H, int T, int d, int b,
                                const void* Z, const float* W_out, const float* aux_out) {
  if (dt != TTT_F32 && dt != TTT_BF16) return TTT_ERR_ARG;
  if (!sizes_ok(B, H, T, d, b)) return TTT_ERR_ARG;
  if (d > kMaxD) return TTT_ERR_UNSUPPORTED;
  const bool needs_rate = variant != ttt::kVarTokenEta, needs_beta = variant == ttt::kVarMomentum;
  const bool needs_tok = variant == ttt::kVarTokenEta;
  const bool needs_v0 = variant == ttt::kVarBias || variant == ttt::kVarLn, needs_v1 = variant == ttt::kVarLn;
  const bool needs_aux = variant == ttt::kVarBias || variant == ttt::kVarMomentum;
  if (!W0 || !W_out || (needs_rate && !rate) || (needs_beta && !mbeta) || (needs_v0 && !vec0) ||
      (needs_v1 && !vec1) || (needs_aux && !aux_out))
    return TTT_ERR_ARG;
  if (T > 0 && (!Q || !K || !V || !Z || (needs_tok && !tok_rate))) return TTT_ERR_ARG;
  for (const void* p : {Q, K, V, static_cast<const void*>(Z), static_cast<const void*>(rate),
                        static_cast<const void*>(mbeta), static_cast<const void*>(tok_rate),
                        static_cast<const void*>(W0), static_cast<const void*>(vec0),
                        static_cast<const void*>(vec1), static_cast<const void*>(W_out),
                        static_cast<const void*>(aux_out)})
    if (p && !aligned16(p)) return TTT_ERR_ARG;
  {
    const size_t seq = bytes4(B, H, T, d, dt == TTT_BF16 ? 2 : 4), hv = bytes4(H, 1, 1, 1, 4);
    const size_t aux = variant == ttt::kVarBias ? bytes4(B, H, d, 1, 4) : bytes4(B, H, d, d, 4);
    if (!outputs_disjoint({{Z, seq}, {W_out, bytes4(B, H, d, d, 4)}, {aux_out, needs_aux ? aux : 0}},
                          {{Q, seq}, {K, seq}, {V, seq}, {rate, needs_rate ? hv : 0}, {mbeta, needs_beta ? hv : 0},
                           {tok_rate, needs_tok ? bytes4(B, H, T, 1, 4) : 0}, {W0, bytes4(H, d, d, 1, 4)},
                           {vec0, needs_v0 ? bytes4(H, d, 1, 1, 4) : 0}, {vec1, needs_v1 ? bytes4(H, d, 1, 1, 4) : 0}}))
      return TTT_ERR_ARG;
  }
  return TTT_OK;
}

static ttt_status variant_simt(int variant, const void* Q, const void* K, const void* V, ttt_dtype dt,
                               const float* rate, const float* mbeta, const float* tok_rate, const float* W0,
                               const float* vec0, const float* vec1, int B, int H, int T, int d, int b, void* Z,
                               float* W_out, float* aux_out, void* stream) {
  ttt::VariantParams p;
  p.Q = Q; p.K = K; p.V = V; p.Z = Z;
  p.rate = rate; p.mbeta = mbeta; p.tok_rate = tok_rate; p.W0 = W0; p.vec0 = vec0; p.vec1 = vec1;
  p.W_out = W_out; p.aux_out = aux_out;
  p.B = B; p.H = H; p.T = T; p.d = d; p.b = b;
  p.units = B * H;
  p.bf16 = dt == TTT_BF16;
  p.variant = variant;
  return ttt::launch_linear_variant(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? TTT_OK : TTT_ERR_CUDA;
}

static ttt_status variant_fwd(int variant, const void* Q, const void* K, const void* V, ttt_dtype dt,
                              const float* rate, const float* mbeta, const float* tok_rate, const float* W0,
                              const float* vec0, const float* vec1, int B, int H, int T, int d, int b, void* Z,
                              float* W_out, float* aux_out, void* stream) {
  const ttt_status st = variant_check(variant, Q, K, V, dt, rate, mbeta, tok_rate, W0, vec0, vec1, B, H, T, d, b, Z,
                                      W_out, aux_out);
  if (st != TTT_OK) return st;
  return variant_simt(variant, Q, K, V, dt, rate, mbeta, tok_rate, W0, vec0, vec1, B, H, T, d, b, Z, W_out, aux_out,
                      stream);
}

// ---------------------------------------------------------------- bias and per-token rate on the
// tensor-core path: the plain rule on changed inputs (linear_prep.cu), padded to 64 features.
namespace {

constexpr int kPadD = 64;

bool variant_fast_ok(int variant, ttt_dtype dt, int d, int b) {
  if (dt != TTT_BF16 || b % 16 != 0) return false;
  if (variant == ttt::kVarBias) return d <= kPadD - 1;
  if (variant == ttt::kVarTokenEta) return d <= kPadD;
  return false;
}

// Byte offsets in the workspace: [status][inner forward's workspace][Q'][K'][V'][Z'][W0'][W_out'][eta'].
// Q', Z' and W_out' exist only when the rows are padded (the bias, or d < 64).
struct VariantLayout {
  size_t sub, sub_bytes, qp, kp, vp, zp, w0p, wp, etap, total;
};

VariantLayout variant_layout(int variant, int B, int H, int T, int d, int b) {
  VariantLayout L{};
  const size_t units = static_cast<size_t>(B) * H;
  const size_t seq = round_up(units * static_cast<size_t>(T) * kPadD * 2, 256);
  const bool pad = variant == ttt::kVarBias || d < kPadD;
  size_t off = kStatusBytes;
  L.sub = off;
  L.sub_bytes = round_up(workspace_bytes_impl(B, H, T, kPadD, b, TTT_VARIANT_LINEAR, nullptr), 256);
  off += L.sub_bytes;
  if (pad) { L.qp = off; off += seq; }
  L.kp = off; off += seq;
  L.vp = off; off += seq;
  if (pad) { L.zp = off; off += seq; }
  L.w0p = off; off += round_up(static_cast<size_t>(H) * kPadD * kPadD * 4, 256);
  if (pad) { L.wp = off; off += round_up(units * kPadD * kPadD * 4, 256); }
  L.etap = off; off += round_up(static_cast<size_t>(H) * 4, 256);
  L.total = off;
  return L;
}

}  // namespace

size_t ttt_linear_variant_workspace_bytes(int variant, ttt_dtype dt, int B, int H, int T, int d, int b) {
  if (!sizes_ok(B, H, T, d, b) || !sizes_ok(B, H, T, kPadD, b)) return 0;
  if (variant == ttt::kVarMomentum || variant == ttt::kVarLn) return kStatusBytes;  // the status word alone
  if (variant != ttt::kVarBias && variant != ttt::kVarTokenEta) return 0;
  if (!variant_fast_ok(variant, dt, d, b)) return kStatusBytes;
  return variant_layout(variant, B, H, T, d, b).total;
}

static ttt_status variant_ex(int variant, const void* Q, const void* K, const void* V, ttt_dtype dt, const float* eta,
                             const float* tok_rate, const float* W0, const float* beta0, int B, int H, int T, int d,
                             int b, void* Z, float* W_out, float* beta_out, void* workspace, size_t ws_bytes,
                             void* stream) {
  ttt_status st = variant_check(variant, Q, K, V, dt, eta, nullptr, tok_rate, W0, beta0, nullptr, B, H, T, d, b, Z,
                                W_out, beta_out);
  if (st != TTT_OK) return st;
  const size_t need = ttt_linear_variant_workspace_bytes(variant, dt, B, H, T, d, b);
  if (need == 0) return TTT_ERR_ARG;
  if (!workspace || !aligned16(workspace) || ws_bytes < need) return TTT_ERR_ARG;
  {
    const size_t seq = bytes4(B, H, T, d, dt == TTT_BF16 ? 2 : 4);
    if (!outputs_disjoint({{Z, seq}, {W_out, bytes4(B, H, d, d, 4)},
                           {beta_out, variant == ttt::kVarBias ? bytes4(B, H, d, 1, 4) : 0}, {workspace, ws_bytes}},
                          {{Q, seq}, {K, seq}, {V, seq}, {eta, variant == ttt::kVarBias ? bytes4(H, 1, 1, 1, 4) : 0},
                           {tok_rate, variant == ttt::kVarTokenEta ? bytes4(B, H, T, 1, 4) : 0},
                           {W0, bytes4(H, d, d, 1, 4)}, {beta0, variant == ttt::kVarBias ? bytes4(H, d, 1, 1, 4) : 0}}))
      return TTT_ERR_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = reset_status(workspace, s);
  if (st != TTT_OK) return st;
  if (!variant_fast_ok(variant, dt, d, b))
    return variant_simt(variant, Q, K, V, dt, eta, nullptr, tok_rate, W0, beta0, nullptr, B, H, T, d, b, Z, W_out,
                        beta_out, stream);

  const VariantLayout L = variant_layout(variant, B, H, T, d, b);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  ttt::VariantPrepParams pp;
  pp.Q = Q; pp.K = K; pp.V = V;
  pp.tok_rate = variant == ttt::kVarTokenEta ? tok_rate : nullptr;
  pp.Qp = L.qp ? ws + L.qp : nullptr;
  pp.Kp = ws + L.kp;
  pp.Vp = ws + L.vp;
  pp.W0 = W0;
  pp.beta0 = variant == ttt::kVarBias ? beta0 : nullptr;
  pp.W0p = reinterpret_cast<float*>(ws + L.w0p);
  pp.eta = variant == ttt::kVarBias ? eta : nullptr;
  pp.etap = reinterpret_cast<float*>(ws + L.etap);
  pp.units = B * H; pp.H = H; pp.T = T; pp.d = d;
  pp.bias = variant == ttt::kVarBias;
  pp.status = static_cast<ttt::StatusBlock*>(workspace);
  if (ttt::launch_variant_prep(pp, s) != cudaSuccess) return TTT_ERR_CUDA;

  void* Zin = L.zp ? static_cast<void*>(ws + L.zp) : Z;
  float* Win = L.wp ? reinterpret_cast<float*>(ws + L.wp) : W_out;
  st = ttt_linear_fwd_ex(pp.Qp ? pp.Qp : Q, pp.Kp, pp.Vp, TTT_BF16, pp.etap, pp.W0p, B, H, T, kPadD, b, Zin, Win,
                         ws + L.sub, L.sub_bytes, stream, nullptr);
  if (st != TTT_OK) return st;

  ttt::VariantPostParams po;
  po.Zp = L.zp ? ws + L.zp : nullptr;
  po.Z = Z;
  po.Wp = L.wp ? reinterpret_cast<const float*>(ws + L.wp) : nullptr;
  po.W_out = W_out;
  po.beta_out = variant == ttt::kVarBias ? beta_out : nullptr;
  po.units = B * H; po.T = T; po.d = d;
  po.status = static_cast<ttt::StatusBlock*>(workspace);
  po.sub = reinterpret_cast<const ttt::StatusBlock*>(ws + L.sub);
  return ttt::launch_variant_post(po, s) == cudaSuccess ? TTT_OK : TTT_ERR_CUDA;
}

ttt_status ttt_linear_bias_fwd_ex(const void* Q, const void* K, const void* V, ttt_dtype dt, const float* eta,
                                  const float* W0, const float* beta0, int B, int H, int T, int d, int b, void* Z,
                                  float* W_out, float* beta_out, void* workspace, size_t ws_bytes, void* stream) {
  return variant_ex(ttt::kVarBias, Q, K, V, dt, eta, nullptr, W0, beta0, B, H, T, d, b, Z, W_out, beta_out, workspace,
                    ws_bytes, stream);
}

ttt_status ttt_linear_token_eta_fwd_ex(const void* Q, const void* K, const void* V, ttt_dtype dt,
                                       const float* eta_tok, const float* W0, int B, int H, int T, int d, int b,
                                       void* Z, float* W_out, void* workspace, size_t ws_bytes, void* stream) {
  return variant_ex(ttt::kVarTokenEta, Q, K, V, dt, nullptr, eta_tok, W0, nullptr, B, H, T, d, b, Z, W_out, nullptr,
                    workspace, ws_bytes, stream);
}

ttt_status ttt_linear_bias_fwd(const void* Q, const void* K, const void* V, ttt_dtype dt, const float* eta,
                               const float* W0, const float* beta0, int B, int H, int T, int d, int b, void* Z,
                               float* W_out, float* beta_out, void* stream) {
  return variant_fwd(ttt::kVarBias, Q, K, V, dt, eta, nullptr, nullptr, W0, beta0, nullptr, B, H, T, d, b, Z, W_out,
                     beta_out, stream);
}

ttt_status ttt_linear_token_eta_fwd(const void* Q, const void* K, const void* V, ttt_dtype dt, const float* eta_tok,
                                    const float* W0, int B, int H, int T, int d, int b, void* Z, float* W_out,
                                    void* stream) {
  return variant_fwd(ttt::kVarTokenEta, Q, K, V, dt, nullptr, nullptr, eta_tok, W0, nullptr, nullptr, B, H, T, d, b,
                     Z, W_out, nullptr, stream);
}

ttt_status ttt_linear_ln_fwd(const void* Q, const void* K, const void* V, ttt_dtype dt, const float* eta,
                             const float* W0, const float* gamma, const float* beta, int B, int H, int T, int d,
                             int b, void* Z, float* W_out, void* stream) {
  return variant_fwd(ttt::kVarLn, Q, K, V, dt, eta, nullptr, nullptr, W0, gamma, beta, B, H, T, d, b, Z, W_out,
                     nullptr, stream);
}

ttt_status ttt_linear_momentum_fwd(const void* Q, const void* K, const void* V, ttt_dtype dt, const float* alpha,
                                   const float* beta, const float* W0, int B, int H, int T, int d, int b, void* Z,
                                   float* W_out, float* M_out, void* stream) {
  return variant_fwd(ttt::kVarMomentum, Q, K, V, dt, alpha, beta, nullptr, W0, nullptr, nullptr, B, H, T, d, b, Z,
                     W_out, M_out, stream);
}

ttt_status ttt_linear_momentum_fwd_ex(const void* Q, const void* K, const void* V, ttt_dtype dt, const float* alpha,
                                      const float* beta, const float* W0, int B, int H, int T, int d, int b, void* Z,
                                      float* W_out, float* M_out, void* workspace, size_t ws_bytes, void* stream,
                                      const ttt_options* opt) {
  ttt_status st = variant_check(ttt::kVarMomentum, Q, K, V, dt, alpha, beta, nullptr, W0, nullptr, nullptr, B, H, T,
                                d, b, Z, W_out, M_out);
  if (st != TTT_OK) return st;
  const size_t need = ttt_linear_variant_workspace_bytes(ttt::kVarMomentum, dt, B, H, T, d, b);
  if (need == 0) return TTT_ERR_ARG;
  if (!workspace || !aligned16(workspace) || ws_bytes < need) return TTT_ERR_ARG;
  const ttt_options o = defaults(opt);
  {
    const size_t seq = bytes4(B, H, T, d, dt == TTT_BF16 ? 2 : 4), dd = bytes4(B, H, d, d, 4);
    if (!outputs_disjoint({{Z, seq}, {W_out, dd}, {M_out, dd}, {workspace, ws_bytes}},
                          {{Q, seq}, {K, seq}, {V, seq}, {alpha, bytes4(H, 1, 1, 1, 4)}, {beta, bytes4(H, 1, 1, 1, 4)},
                           {W0, bytes4(H, d, d, 1, 4)}}))
      return TTT_ERR_ARG;
  }
  if (o.force_path < 0 || o.force_path > 3) return TTT_ERR_ARG;
  const bool mma = ttt::linear_mom_mma_supported(d, b, dt == TTT_BF16) && T > 0;
  if (o.force_path == 3 || (o.force_path == 2 && !mma)) return TTT_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = reset_status(workspace, s);
  if (st != TTT_OK) return st;
  if (!mma || o.force_path == 1)
    return variant_simt(ttt::kVarMomentum, Q, K, V, dt, alpha, beta, nullptr, W0, nullptr, nullptr, B, H, T, d, b, Z,
                        W_out, M_out, stream);
  ttt::MomParams p;
  p.Q = Q; p.K = K; p.V = V; p.Z = Z;
  p.alpha = alpha; p.beta = beta; p.W0 = W0; p.W_out = W_out; p.M_out = M_out;
  p.H = H; p.T = T; p.b = b; p.units = B * H;
  p.status = static_cast<ttt::StatusBlock*>(workspace);
  p.timeout_ns = o.wait_timeout_ns;
  p.inject_stall = o.inject_stall;
  CUtensorMap mq, mk, mv;
  const int rows = ttt::linear_mom_mma_tile_rows();
  if (!encode_3d(&mq, Q, p.units, T, d, rows, d, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_3d(&mk, K, p.units, T, d, rows, d, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_3d(&mv, V, p.units, T, d, rows, d, CU_TENSOR_MAP_SWIZZLE_128B))
    return TTT_ERR_CUDA;
  return ttt::launch_linear_mom_mma(p, mq, mk, mv, s) == cudaSuccess ? TTT_OK : TTT_ERR_CUDA;
}

ttt_status ttt_linear_ln_fwd_ex(const void* Q, const void* K, const void* V, ttt_dtype dt, const float* eta,
                                const float* W0, const float* gamma, const float* beta, int B, int H, int T, int d,
                                int b, void* Z, float* W_out, void* workspace, size_t ws_bytes, void* stream,
                                const ttt_options* opt) {
  ttt_status st = variant_check(ttt::kVarLn, Q, K, V, dt, eta, nullptr, nullptr, W0, gamma, beta, B, H, T, d, b, Z,
                                W_out, nullptr);
  if (st != TTT_OK) return st;
  const size_t need = ttt_linear_variant_workspace_bytes(ttt::kVarLn, dt, B, H, T, d, b);
  if (need == 0) return TTT_ERR_ARG;
  if (!workspace || !aligned16(workspace) || ws_bytes < need) return TTT_ERR_ARG;
  const ttt_options o = defaults(opt);
  {
    const size_t seq = bytes4(B, H, T, d, dt == TTT_BF16 ? 2 : 4), hd = bytes4(H, d, 1, 1, 4);
    if (!outputs_disjoint({{Z, seq}, {W_out, bytes4(B, H, d, d, 4)}, {workspace, ws_bytes}},
                          {{Q, seq}, {K, seq}, {V, seq}, {eta, bytes4(H, 1, 1, 1, 4)}, {W0, bytes4(H, d, d, 1, 4)},
                           {gamma, hd}, {beta, hd}}))
      return TTT_ERR_ARG;
  }
  if (o.force_path < 0 || o.force_path > 3) return TTT_ERR_ARG;
  const bool mma = ttt::linear_ln_mma_supported(d, b, dt == TTT_BF16) && T > 0;
  if (o.force_path == 3 || (o.force_path == 2 && !mma)) return TTT_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = reset_status(workspace, s);
  if (st != TTT_OK) return st;
  if (!mma || o.force_path == 1)
    return variant_simt(ttt::kVarLn, Q, K, V, dt, eta, nullptr, nullptr, W0, gamma, beta, B, H, T, d, b, Z, W_out,
                        nullptr, stream);
  ttt::LnParams p;
  p.Q = Q; p.K = K; p.V = V; p.Z = Z;
  p.eta = eta; p.gamma = gamma; p.beta = beta; p.W0 = W0; p.W_out = W_out;
  p.H = H; p.T = T; p.b = b; p.units = B * H;
  p.status = static_cast<ttt::StatusBlock*>(workspace);
  p.timeout_ns = o.wait_timeout_ns;
  p.inject_stall = o.inject_stall;
  CUtensorMap mq, mk, mv;
  const int rows = ttt::linear_ln_mma_tile_rows();
  if (!encode_3d(&mq, Q, p.units, T, d, rows, d, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_3d(&mk, K, p.units, T, d, rows, d, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_3d(&mv, V, p.units, T, d, rows, d, CU_TENSOR_MAP_SWIZZLE_128B))
    return TTT_ERR_CUDA;
  return ttt::launch_linear_ln_mma(p, mq, mk, mv, s) == cudaSuccess ? TTT_OK : TTT_ERR_CUDA;
}

// Segments of the tensor-core backward (bf16, d = 64, b = 16): as many as fill the SMs with one
// CTA per (unit, segment), each a whole number of 64-token blocks.
struct BwdPlan {
  int seg_len, seg_count;
};

BwdPlan plan_linear_bwd(int B, int H, int T, int d, int b, bool mma) {
  BwdPlan pl{static_cast<int>(round_up(static_cast<size_t>(T > 0 ? T : 1), 64)), 1};
  if (!mma || T <= 64 || d != 64 || b != 16) return pl;
  const long long units = static_cast<long long>(B) * H;
  const long long want = std::min<long long>((T + 63) / 64, std::max<long long>(1, sm_count() / units));
  if (want < 2) return pl;
  const long long len = round_up(static_cast<size_t>((T + want - 1) / want), 64);
  pl.seg_len = static_cast<int>(len);
  pl.seg_count = static_cast<int>((T + len - 1) / len);
  return pl;
}

// Bytes after the backward's states and partials: per-segment partials, the forward's segment
// maps and start states, H_s and A_s, the segments' end gradients (fp32).
size_t bwd_seg_bytes(const BwdPlan& pl, int units) {
  if (pl.seg_count < 2) return 0;
  const size_t dd = 64 * 64, u = static_cast<size_t>(units), S = pl.seg_count;
  return round_up(u * S * (dd + 1) * 4, 256) + u * (S - 1) * dd * 4 * (2 + 1 + 2 + 1);
}

size_t ttt_linear_bwd_workspace_bytes(int B, int H, int T, int d, int b) {
  if (!sizes_ok(B, H, T, d, b)) return 0;
  // Sized for bf16 operands, the only dtype whose backward may use segments.
  const BwdPlan pl = plan_linear_bwd(B, H, T, d, b, ttt::linear_bwd_mma_supported(d, b, true) && T > 0);
  return kStatusBytes + round_up(ttt::linear_bwd_scratch_bytes(B * H, T, d, b), 16) + bwd_seg_bytes(pl, B * H);
}

ttt_status ttt_linear_bwd(const void* Q, const void* K, const void* V, ttt_dtype dt, const float* eta,
                          const float* W0, int B, int H, int T, int d, int b, const void* dZ, const float* dW_out,
                          void* dQ, void* dK, void* dV, float* deta, float* dW0, void* workspace, size_t ws_bytes,
                          void* stream) {
  if (dt != TTT_F32 && dt != TTT_BF16) return TTT_ERR_ARG;
  if (!sizes_ok(B, H, T, d, b)) return TTT_ERR_ARG;
  const bool bf16 = dt == TTT_BF16;
  const bool mma = ttt::linear_bwd_mma_supported(d, b, bf16) && T > 0;
  if (!mma && !ttt::linear_bwd_supported(d, b)) return TTT_ERR_UNSUPPORTED;
  if (!eta || !W0 || !dW_out || !deta || !dW0 || !workspace) return TTT_ERR_ARG;
  if (T > 0 && (!Q || !K || !V || !dZ || !dQ || !dK || !dV)) return TTT_ERR_ARG;
  for (const void* p : {Q, K, V, dZ, static_cast<const void*>(dQ), static_cast<const void*>(dK),
                        static_cast<const void*>(dV), static_cast<const void*>(eta), static_cast<const void*>(W0),
                        static_cast<const void*>(dW_out), static_cast<const void*>(deta),
                        static_cast<const void*>(dW0), static_cast<const void*>(workspace)})
    if (p && !aligned16(p)) return TTT_ERR_ARG;
  if (ws_bytes < ttt_linear_bwd_workspace_bytes(B, H, T, d, b)) return TTT_ERR_ARG;
  {
    const size_t seq = bytes4(B, H, T, d, bf16 ? 2 : 4), hdd = bytes4(H, d, d, 1, 4);
    if (!outputs_disjoint({{dQ, seq}, {dK, seq}, {dV, seq}, {deta, bytes4(H, 1, 1, 1, 4)}, {dW0, hdd},
                           {workspace, ws_bytes}},
                          {{Q, seq}, {K, seq}, {V, seq}, {dZ, seq}, {eta, bytes4(H, 1, 1, 1, 4)}, {W0, hdd},
                           {dW_out, bytes4(B, H, d, d, 4)}}))
      return TTT_ERR_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ttt::LinearBwdParams p;
  p.Q = Q; p.K = K; p.V = V; p.dZ = dZ;
  p.eta = eta;
  p.W0 = W0;
  p.dW_out = dW_out;
  p.dQ = dQ; p.dK = dK; p.dV = dV;
  p.deta = deta;
  p.dW0 = dW0;
  p.B = B; p.H = H; p.T = T; p.d = d; p.b = b;
  p.units = B * H;
  p.bf16 = bf16;
  p.states = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + kStatusBytes);
  const size_t nch = (static_cast<size_t>(T) + b - 1) / b;
  p.partial = p.states + static_cast<size_t>(p.units) * nch * d * d;
  p.chunk_buf = ttt::linear_bwd_chunk_buf(p.partial, p.units, d);
  p.status = static_cast<ttt::StatusBlock*>(workspace);
  const BwdPlan bpl = plan_linear_bwd(B, H, T, d, b, mma);
  p.bseg_len = bpl.seg_len;
  p.bseg_count = bpl.seg_count;
  p.w_starts = nullptr;
  p.hA = nullptr;
  p.g_ends = nullptr;
  float* seg_maps = nullptr;
  float* seg_starts = nullptr;
  if (bpl.seg_count > 1) {
    const size_t dd = static_cast<size_t>(d) * d, S = bpl.seg_count, u = p.units;
    uint8_t* seg = static_cast<uint8_t*>(workspace) + kStatusBytes +
                   round_up(ttt::linear_bwd_scratch_bytes(B * H, T, d, b), 16);
    p.partial = reinterpret_cast<float*>(seg);
    seg_maps = reinterpret_cast<float*>(seg + round_up(u * S * (dd + 1) * 4, 256));
    seg_starts = seg_maps + u * (S - 1) * 2 * dd;
    p.hA = seg_starts + u * (S - 1) * dd;
    p.g_ends = p.hA + u * (S - 1) * 2 * dd;
    p.w_starts = seg_starts;
  }
  p.timeout_ns = kDefaultTimeoutNs;
  const ttt_status st = reset_status(workspace, s);
  if (st != TTT_OK) return st;
  cudaError_t err;
  if (mma) {
    CUtensorMap mq, mk, mv, mdz;
    const int rows = ttt::linear_bwd_mma_rows();
    if (!encode_3d(&mq, Q, p.units, T, d, rows, d, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_3d(&mk, K, p.units, T, d, rows, d, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_3d(&mv, V, p.units, T, d, rows, d, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_3d(&mdz, dZ, p.units, T, d, rows, d, CU_TENSOR_MAP_SWIZZLE_128B))
      return TTT_ERR_CUDA;
    err = cudaSuccess;
    if (bpl.seg_count > 1) {
      // Start states of segments 1..S-1: the forward's segment maps and their combine.
      ttt::LinearParams fp{};
      fp.Q = Q; fp.K = K; fp.V = V; fp.Z = nullptr;
      fp.eta = eta; fp.W0 = W0; fp.W_out = nullptr;
      fp.B = B; fp.H = H; fp.T = T; fp.d = d; fp.b = b;
      fp.units = p.units;
      fp.bf16 = true;
      fp.status = p.status;
      fp.timeout_ns = p.timeout_ns;
      fp.inject_stall = 0;
      fp.seg_len = bpl.seg_len;
      fp.seg_count = bpl.seg_count;
      fp.seg_maps = seg_maps;
      fp.seg_starts = seg_starts;
      fp.affine_wy = 1;
      fp.seg_first = 0;
      fp.seg_num = bpl.seg_count - 1;
      CUtensorMap mk64, mv64, mq16, mk16, mdz16;
      const int rows64 = ttt::linear_seg_wy_rows(), rows16 = ttt::linear_bwd_hmap_rows();
      if (!encode_3d(&mk64, K, p.units, T, d, rows64, d, CU_TENSOR_MAP_SWIZZLE_128B) ||
          !encode_3d(&mv64, V, p.units, T, d, rows64, d, CU_TENSOR_MAP_SWIZZLE_128B) ||
          !encode_3d(&mq16, Q, p.units, T, d, rows16, d, CU_TENSOR_MAP_SWIZZLE_128B) ||
          !encode_3d(&mk16, K, p.units, T, d, rows16, d, CU_TENSOR_MAP_SWIZZLE_128B) ||
          !encode_3d(&mdz16, dZ, p.units, T, d, rows16, d, CU_TENSOR_MAP_SWIZZLE_128B))
        return TTT_ERR_CUDA;
      err = ttt::launch_linear_seg_affine_wy(fp, mk64, mv64, s);
      if (err == cudaSuccess) err = ttt::launch_linear_seg_combine(fp, s);
      // H_s, A_s of segments 1..S-1 and the gradients at the segments' ends.
      if (err == cudaSuccess) err = ttt::launch_linear_bwd_hmap(p, mq16, mk16, mdz16, s);
      if (err == cudaSuccess) err = ttt::launch_linear_bwd_rcombine(p, s);
    }
    if (err == cudaSuccess) err = ttt::launch_linear_bwd_mma(p, mq, mk, mv, mdz, s);
  } else {
    err = ttt::launch_linear_bwd(p, s);
  }
  if (err == cudaSuccess) err = ttt::launch_linear_bwd_reduce(p, s);
  return err == cudaSuccess ? TTT_OK : TTT_ERR_CUDA;
}

size_t ttt_mlp_bwd_workspace_bytes(int B, int H, int T, int d, int b) {
  if (!sizes_ok(B, H, T, d, b)) return 0;
  return kStatusBytes + round_up(ttt::mlp_bwd_scratch_bytes(B * H, T, d, b), 16);
}

ttt_status ttt_mlp_bwd(const void* Q, const void* K, const void* V, ttt_dtype dt, const float* eta,
                       const float* W1_0, const float* W2_0, int B, int H, int T, int d, int b, const void* dZ,
                       const float* dW1_out, const float* dW2_out, void* dQ, void* dK, void* dV, float* deta,
                       float* dW1, float* dW2, void* workspace, size_t ws_bytes, void* stream) {
  if (dt != TTT_F32 && dt != TTT_BF16) return TTT_ERR_ARG;
  if (!sizes_ok(B, H, T, d, b)) return TTT_ERR_ARG;
  if (d > kMaxD) return TTT_ERR_UNSUPPORTED;
  if (!eta || !W1_0 || !W2_0 || !dW1_out || !dW2_out || !deta || !dW1 || !dW2 || !workspace) return TTT_ERR_ARG;
  if (T > 0 && (!Q || !K || !V || !dZ || !dQ || !dK || !dV)) return TTT_ERR_ARG;
  for (const void* p : {Q, K, V, dZ, static_cast<const void*>(dQ), static_cast<const void*>(dK),
                        static_cast<const void*>(dV), static_cast<const void*>(eta), static_cast<const void*>(W1_0),
                        static_cast<const void*>(W2_0), static_cast<const void*>(dW1_out),
                        static_cast<const void*>(dW2_out), static_cast<const void*>(deta),
                        static_cast<const void*>(dW1), static_cast<const void*>(dW2),
                        static_cast<const void*>(workspace)})
    if (p && !aligned16(p)) return TTT_ERR_ARG;
  if (ws_bytes < ttt_mlp_bwd_workspace_bytes(B, H, T, d, b)) return TTT_ERR_ARG;
  const int m = static_cast<int>(mlp_hidden(d));
  {
    const size_t seq = bytes4(B, H, T, d, dt == TTT_BF16 ? 2 : 4), hw = bytes4(H, d, m, 1, 4);
    const size_t bw = bytes4(B, H, d, m, 4);
    if (!outputs_disjoint({{dQ, seq}, {dK, seq}, {dV, seq}, {deta, bytes4(H, 1, 1, 1, 4)}, {dW1, hw}, {dW2, hw},
                           {workspace, ws_bytes}},
                          {{Q, seq}, {K, seq}, {V, seq}, {dZ, seq}, {eta, bytes4(H, 1, 1, 1, 4)}, {W1_0, hw},
                           {W2_0, hw}, {dW1_out, bw}, {dW2_out, bw}}))
      return TTT_ERR_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ttt::MlpBwdParams p;
  p.Q = Q; p.K = K; p.V = V; p.dZ = dZ;
  p.eta = eta; p.W1_0 = W1_0; p.W2_0 = W2_0; p.dW1_out = dW1_out; p.dW2_out = dW2_out;
  p.dQ = dQ; p.dK = dK; p.dV = dV;
  p.deta = deta; p.dW1 = dW1; p.dW2 = dW2;
  p.B = B; p.H = H; p.T = T; p.d = d; p.m = m; p.b = b;
  p.units = B * H;
  p.bf16 = dt == TTT_BF16;
  p.scratch = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + kStatusBytes);
  p.partial = p.scratch + static_cast<size_t>(p.units) * ttt::mlp_bwd_unit_floats(T, d, b);
  const ttt_status st = reset_status(workspace, s);
  if (st != TTT_OK) return st;
  return ttt::launch_mlp_bwd(p, s) == cudaSuccess ? TTT_OK : TTT_ERR_CUDA;
}

ttt_status ttt_last_device_status(void* workspace, void* stream) {
  if (!workspace || !aligned16(workspace)) return TTT_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ttt::StatusBlock host;
  if (cudaMemcpyAsync(&host, workspace, sizeof(host), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return TTT_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return TTT_ERR_CUDA;
  if (cudaMemsetAsync(workspace, 0, sizeof(host), s) != cudaSuccess) return TTT_ERR_CUDA;
  if (host.code == 0) return TTT_OK;
  return static_cast<ttt_status>(host.code);
}

}  // extern "C"
