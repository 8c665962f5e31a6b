// Launch interface between the C ABI (ttt_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ttt.h"

namespace ttt {

struct StatusBlock;

struct LinearParams {
  const void* Q;
  const void* K;
  const void* V;
  void* Z;
  const float* eta;    // [H]
  const float* W0;     // [H][d][d]
  float* W_out;        // [B][H][d][d]
  int B, H, T, d, b;
  int units;           // B * H
  bool bf16;           // Q, K, V, Z are bf16 (else fp32)
  StatusBlock* status;
  uint64_t timeout_ns;
  int inject_stall;
  // Segment-parallel form (tensor-core path only). seg_count == 1: one pass
  // over the whole sequence. Otherwise the sequence is cut into seg_count
  // segments of seg_len tokens (a multiple of b and of 16; the last may be
  // shorter) that run side by side from start states the combine step computes.
  int seg_len;
  int seg_count;
  // The segments one launch covers: [seg_first, seg_first + seg_num) (segments
  // for the read-out, maps for the affine and combine kernels). A call may
  // split the range over several launches so that the affine maps of later
  // segments overlap the read-out of earlier ones.
  int seg_first;
  int seg_num;
  float* seg_maps;     // workspace [units][seg_count-1][2][d][d]: (A_s, B_s)
  float* seg_starts;   // workspace [units][seg_count-1][d][d]: start state of segment s+1
  int affine_wy;       // affine maps on the tcgen05 kernel (64-token steps); else warp-level MMAs
};

struct MlpParams {
  const void* Q;
  const void* K;
  const void* V;
  void* Z;
  const float* eta;
  const float* W1_0;   // [H][d][m]
  const float* W2_0;   // [H][m][d]
  float* W1_out;       // [B][H][d][m]  (running state while the kernel works)
  float* W2_out;       // [B][H][m][d]
  float* snap;         // workspace: per unit d*m + m*d floats (chunk-start snapshot)
  int B, H, T, d, m, b;
  int units;
  bool bf16;
  StatusBlock* status;
  uint64_t timeout_ns;
  int inject_stall;
};

// Backward of TTT-Linear: upstream dZ, dW_out -> dQ, dK, dV (the dtype of Q),
// d eta [H] and dW0 [H][d][d] (summed over batch rows).
struct LinearBwdParams {
  const void* Q;
  const void* K;
  const void* V;
  const void* dZ;
  const float* eta;
  const float* W0;
  const float* dW_out;
  void* dQ;
  void* dK;
  void* dV;
  float* deta;
  float* dW0;
  int B, H, T, d, b;
  int units;
  bool bf16;       // Q, K, V, dZ, dQ, dK, dV are bf16 (else fp32)
  float* states;   // workspace [units][ceil(T/b)][d][d]: chunk-start states (tensor-core kernel:
                   // the state at the start of every 64-token block)
  float* partial;  // workspace [units][d*d + 1]: per-unit dW0, then d eta
  float* chunk_buf;  // workspace [units][2][min(b, T)][d]: E, dE of one chunk (chunks longer than 64)
  // Segments (tensor-core kernel): a unit's sequence in bseg_count ranges of bseg_len tokens (a
  // multiple of 64), one CTA each; partial is then [units][bseg_count][d*d + 1].
  int bseg_len;
  int bseg_count;
  const float* w_starts;  // [units][S-1][d][d]: W at the start of segments 1..S-1
  float* hA;              // [units][S-1][2][d][d]: H_s, then A_s, of segments 1..S-1
  float* g_ends;          // [units][S-1][d][d]: gradient of the end state of segments 0..S-2
  StatusBlock* status;
  uint64_t timeout_ns;
};

// Backward of TTT-MLP (mlp_bwd.cu), fp32 arithmetic, d <= 64, hidden m = 4d, any b.
struct MlpBwdParams {
  const void* Q;
  const void* K;
  const void* V;
  const void* dZ;
  const float* eta;
  const float* W1_0;     // [H][d][m]
  const float* W2_0;     // [H][m][d]
  const float* dW1_out;  // [B][H][d][m]
  const float* dW2_out;  // [B][H][m][d]
  void* dQ;
  void* dK;
  void* dV;
  float* deta;           // [H]
  float* dW1;            // [H][d][m]
  float* dW2;            // [H][m][d]
  int B, H, T, d, m, b;
  int units;
  bool bf16;             // Q, K, V, dZ, dQ, dK, dV are bf16 (else fp32)
  float* scratch;        // workspace [units][mlp_bwd_unit_floats]
  float* partial;        // workspace [units][2 d m + 1]
};
// Floats of one unit's scratch: chunk-start weights, the gradient accumulators and
// one chunk's matrices.
__host__ __device__ inline size_t mlp_bwd_unit_floats(int T, int d, int b) {
  const size_t m = static_cast<size_t>(4) * d, dm = static_cast<size_t>(d) * m;
  const size_t nch = (static_cast<size_t>(T) + b - 1) / b;
  const size_t cap = static_cast<size_t>(T < b ? T : b);
  return nch * 2 * dm + 4 * dm + 8 * cap * d + 11 * cap * m + 3 * cap * cap;
}
size_t mlp_bwd_scratch_bytes(int units, int T, int d, int b);  // scratch + partials
cudaError_t launch_mlp_bwd(const MlpBwdParams& p, cudaStream_t stream);  // both kernels

// Inner-model variants of TTT-Linear (linear_variants.cu), fp32 arithmetic.
enum : int { kVarBias = TTT_INNER_BIAS, kVarTokenEta = TTT_INNER_TOKEN_ETA, kVarLn = TTT_INNER_LN,
              kVarMomentum = TTT_INNER_MOMENTUM };
struct VariantParams {
  const void* Q;
  const void* K;
  const void* V;
  void* Z;
  const float* rate;      // [H]: eta (bias, LN) or alpha (momentum); unused for per-token rates
  const float* mbeta;     // [H]: momentum coefficient beta (momentum only)
  const float* tok_rate;  // [B][H][T]: per-token learning rate (per-token variant only)
  const float* W0;        // [H][d][d]
  const float* vec0;      // [H][d]: beta0 (bias) or gamma (LN)
  const float* vec1;      // [H][d]: beta (LN)
  float* W_out;           // [B][H][d][d]
  float* aux_out;         // [B][H][d] final bias, or [B][H][d][d] final momentum
  int B, H, T, d, b;
  int units;
  bool bf16;
  int variant;            // kVar*
};
cudaError_t launch_linear_variant(const VariantParams& p, cudaStream_t stream);

// The momentum variant on the tensor cores (linear_mom_mma.cu): bf16, d = 64, b % 16 = 0,
// one CTA per (batch row, head).
struct MomParams {
  const void* Q;          // [units][T][64] bf16
  const void* K;
  const void* V;
  void* Z;
  const float* alpha;     // [H]
  const float* beta;      // [H]
  const float* W0;        // [H][64][64]
  float* W_out;           // [units][64][64]
  float* M_out;           // [units][64][64]
  int H, T, b, units;
  StatusBlock* status;
  uint64_t timeout_ns;
  int inject_stall;
};
bool linear_mom_mma_supported(int d, int b, bool bf16);
int linear_mom_mma_tile_rows();
cudaError_t launch_linear_mom_mma(const MomParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                                  const CUtensorMap& mv, cudaStream_t stream);

// The layer-norm + residual variant on the tensor cores (linear_ln_mma.cu): bf16, d = 64,
// b % 16 = 0, one CTA per (batch row, head).
struct LnParams {
  const void* Q;          // [units][T][64] bf16
  const void* K;
  const void* V;
  void* Z;
  const float* eta;       // [H]
  const float* gamma;     // [H][64]
  const float* beta;      // [H][64]
  const float* W0;        // [H][64][64]
  float* W_out;           // [units][64][64]
  int H, T, b, units;
  StatusBlock* status;
  uint64_t timeout_ns;
  int inject_stall;
};
bool linear_ln_mma_supported(int d, int b, bool bf16);
int linear_ln_mma_tile_rows();
cudaError_t launch_linear_ln_mma(const LnParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                                 const CUtensorMap& mv, cudaStream_t stream);

// The bias and per-token-rate variants as the plain rule on changed inputs
// (linear_prep.cu): padded to 64 features, bf16.
struct VariantPrepParams {
  const void* Q;            // [units][T][d] bf16
  const void* K;
  const void* V;
  const float* tok_rate;    // [units][T] (per-token rate; null: none)
  void* Qp;                 // [units][T][64] bf16; null: Q is used as it is
  void* Kp;
  void* Vp;
  const float* W0;          // [H][d][d]
  const float* beta0;       // [H][d] (bias)
  float* W0p;               // [H][64][64]
  const float* eta;         // [H]; null: ones
  float* etap;              // [H]
  int units, H, T, d;
  bool bias;
  StatusBlock* status;
};
cudaError_t launch_variant_prep(const VariantPrepParams& p, cudaStream_t stream);

struct VariantPostParams {
  const void* Zp;           // [units][T][64] bf16; null: Z was written in place
  void* Z;                  // [units][T][d] bf16
  const float* Wp;          // [units][64][64]; null: W_out was written in place
  float* W_out;             // [units][d][d]
  float* beta_out;          // [units][d] (bias) or null
  int units, T, d;
  StatusBlock* status;      // the call's status word
  const StatusBlock* sub;   // the inner forward's
};
cudaError_t launch_variant_post(const VariantPostParams& p, cudaStream_t stream);

struct DecodeParams {
  const void* q;
  const void* k;
  const void* v;
  void* z;
  const float* eta;
  float* W_anchor;
  float* W_run;
  int B, H, d, pos, b;
  int N;               // tokens per (batch row, head); q, k, v, z are [B][H][N][d]
  int units;
  bool bf16;
};

// Tensor-core TTT-Linear (bf16, d = 64, b % 16 == 0).
bool linear_mma_supported(const LinearParams& p);
int linear_mma_tile_rows();
cudaError_t launch_linear_mma(const LinearParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                              const CUtensorMap& mv, cudaStream_t stream);

// Segment-parallel TTT-Linear (bf16, d = 64, b % 16 == 0): per-segment affine
// maps, then the combine over segments; linear_mma then runs every segment.
bool linear_seg_supported(const LinearParams& p);
cudaError_t launch_linear_seg_affine(const LinearParams& p, const CUtensorMap& mk, const CUtensorMap& mv,
                                     cudaStream_t stream);
cudaError_t launch_linear_seg_combine(const LinearParams& p, cudaStream_t stream);
// The affine maps on tcgen05 in 64-token steps (b = 16, 32 or a multiple of 64;
// seg_len a multiple of 64 and of b). Tensor maps with 64-row boxes.
bool linear_seg_wy_supported(int b, int seg_len);
int linear_seg_wy_rows();
cudaError_t launch_linear_seg_affine_wy(const LinearParams& p, const CUtensorMap& mk64, const CUtensorMap& mv64,
                                        cudaStream_t stream);

// General fp32-arithmetic TTT-Linear (any dtype, d <= 64, any b).
cudaError_t launch_linear_simt(const LinearParams& p, cudaStream_t stream);

// Tensor-core TTT-MLP (bf16, d = 64, hidden 256, b % 16 == 0), one CTA per unit.
bool mlp_mma_supported(const MlpParams& p);
bool mlp_cluster_supported(const MlpParams& p);  // b = 16: two CTAs per unit (mlp_cluster.cu)
cudaError_t launch_mlp_cluster(const MlpParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                               const CUtensorMap& mv, cudaStream_t stream);
int mlp_mma_tile_rows();
cudaError_t launch_mlp_mma(const MlpParams& p, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                           cudaStream_t stream);

// The TTT-MLP forward behind ttt_mlp_fwd(_ex) and ttt_mlp_fwd_noalloc (ttt_api.cu):
// argument checks, workspace layout and launch. With ws_by_path the workspace
// need only cover the kernel that serves the call (mlp_workspace_bytes_for_path);
// otherwise it must cover ttt_workspace_bytes(), which sizes for every kernel.
ttt_status mlp_forward(const void* Q, const void* K, const void* V, ttt_dtype dt, const float* eta,
                       const float* W1_0, const float* W2_0, int B, int H, int T, int d, int b, void* Z,
                       float* W1_out, float* W2_out, void* workspace, size_t ws_bytes, void* stream,
                       const ttt_options* opt, bool ws_by_path);
// Whether the tensor-core kernel serves such a call (it keeps the chunk-start
// weights on chip and uses only the status block of the workspace).
bool mlp_uses_mma(int T, int d, int b, ttt_dtype dt, const ttt_options* opt);
// Workspace bytes the kernel that serves such a call uses (0 for invalid sizes).
size_t mlp_workspace_bytes_for_path(int B, int H, int T, int d, int b, ttt_dtype dt, const ttt_options* opt);

// General fp32-arithmetic TTT-MLP.
size_t mlp_simt_snapshot_bytes(int units, int d, int m);
cudaError_t launch_mlp_simt(const MlpParams& p, cudaStream_t stream);

// Decode token.
cudaError_t launch_linear_decode(const DecodeParams& p, cudaStream_t stream);

// Backward of TTT-Linear in fp32 arithmetic, fp32 or bf16 operands, d <= 64, b <= 64
// (linear_bwd.cu), and the sum of the per-unit dW0, d eta shares over batch rows.
bool linear_bwd_supported(int d, int b);
size_t linear_bwd_smem_bytes(int d, int b);
size_t linear_bwd_scratch_bytes(int units, int T, int d, int b);  // states + partials, bytes
float* linear_bwd_chunk_buf(float* partial, int units, int d);       // where chunk_buf starts
cudaError_t launch_linear_bwd(const LinearBwdParams& p, cudaStream_t stream);
cudaError_t launch_linear_bwd_reduce(const LinearBwdParams& p, cudaStream_t stream);
// Segment-parallel backward (linear_bwd_seg.cu): H_s and A_s of segments 1..S-1, and the
// gradients at the segments' ends.
int linear_bwd_hmap_rows();
cudaError_t launch_linear_bwd_hmap(const LinearBwdParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                                   const CUtensorMap& mdz, cudaStream_t stream);
cudaError_t launch_linear_bwd_rcombine(const LinearBwdParams& p, cudaStream_t stream);

// Backward of TTT-Linear on the tensor cores (linear_bwd_mma.cu): bf16, d = 64, b = 16.
// Tensor maps over Q, K, V, dZ with linear_bwd_mma_rows()-row boxes.
bool linear_bwd_mma_supported(int d, int b, bool bf16);
int linear_bwd_mma_rows();
cudaError_t launch_linear_bwd_mma(const LinearBwdParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                                  const CUtensorMap& mv, const CUtensorMap& mdz, cudaStream_t stream);

}  // namespace ttt
