// Inner-model variants of TTT-Linear, fp32 arithmetic, any d <= 64, any chunk
// size b, fp32 or bf16 inputs. One CTA per (batch row, head); the state lives in
// shared memory; a chunk is walked in pieces of at most 16 tokens that never
// cross a chunk boundary (as linear_simt.cu does for the plain layer).
//
// The variants and where they come from (the pages name them; the formulas are
// the readings stated in include/ttt.h beside each entry point):
//   - bias: f(k) = k W + beta ("Test-Time Training (TTT) guide", section 3,
//     f(W, x) = W x + b). With e = k W_a + beta_a - v, W -= eta k^T e and
//     beta -= eta e; read-out q W + beta. Within a piece the read-out weight of
//     token i for token t is (q_t . k_i + 1): the bias is a constant extra input.
//   - per-token learning rate ("5 · TestingTime 训练与长上下文", section 3.1, a
//     learnable learning rate): token i's gradient is scaled by eta_i, so its
//     read-out weight becomes eta_i (q_t . k_i) and the update sums eta_i k_i^T e_i.
//   - layer norm and residual inside f (same page, section 3.1): f(k) = k + LN(k W);
//     the error is the chain rule through LN, e = (g - mean(g) - x mean(g x)) / s
//     with y = k W_a, x = (y - mean y) / s, g = gamma (k + gamma x + beta - v);
//     read-out z = q + LN(q W_a - eta tril(q K^T) E) (the chunk's dual form).
//   - momentum ("推理时的“临阵磨枪”：Test-Time Training如何教会AI“边做边学”",
//     sections 2.3 and 5.1): per token, with chunk-start gradients g_t =
//     k_t^T (k_t W_a - v_t), M <- beta M + (1 - beta) g_t and W <- W - alpha M.
//     From the running (W, M) at a piece start, token t of the piece (1-based)
//     reads out z_t = q_t W - alpha c_t (q_t M) - alpha sum_{i <= t}
//     (1 - beta^(t-i+1)) (q_t . k_i) e_i with c_t = beta + ... + beta^t, and after
//     the piece's n tokens W -= alpha (c_n M + sum_i (1 - beta^(n-i+1)) k_i^T e_i),
//     M = beta^n M + (1 - beta) sum_i beta^(n-i) k_i^T e_i (the closed form of the
//     recurrence; M is not reset at chunk boundaries).
#include "kernels.h"
#include "ttt_device.cuh"

namespace ttt {
namespace {

constexpr int kPiece = 16;
constexpr int kThreads = 256;
constexpr int kWarpsV = kThreads / 32;
constexpr float kLnEps = 1e-6f;

template <typename T>
__device__ __forceinline__ float ld_in(const T* p);
template <>
__device__ __forceinline__ float ld_in<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ld_in<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }

template <typename T>
__device__ __forceinline__ void st_out(T* p, float v);
template <>
__device__ __forceinline__ void st_out<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void st_out<__nv_bfloat16>(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Row-wise layer norm of the n rows of X [n][d] in place: X <- x (the normalised
// row, gamma and beta not applied); rs[t] <- 1 / s_t. One warp per row.
__device__ void normalise_rows(float* X, float* rs, int n, int d, int warp, int lane) {
  for (int t = warp; t < n; t += kWarpsV) {
    float* row = X + t * d;
    float sum = 0.f;
    for (int j = lane; j < d; j += 32) sum += row[j];
    const float mu = warp_sum(sum) / d;
    float sq = 0.f;
    for (int j = lane; j < d; j += 32) {
      const float c = row[j] - mu;
      sq += c * c;
    }
    const float inv = rsqrtf(warp_sum(sq) / d + kLnEps);
    for (int j = lane; j < d; j += 32) row[j] = (row[j] - mu) * inv;
    if (lane == 0) rs[t] = inv;
  }
}

template <typename T, int kVar>
__global__ void __launch_bounds__(kThreads) linear_variant_kernel(VariantParams p) {
  extern __shared__ float sm[];
  const int d = p.d;
  float* Wr = sm;                // running W [d][d]
  float* Wa = Wr + d * d;        // chunk-start W [d][d]
  float* Mr = Wa + d * d;        // running momentum [d][d] (momentum only)
  float* Qs = Mr + (kVar == kVarMomentum ? d * d : 0);  // [16][d]
  float* Ks = Qs + kPiece * d;
  float* Vs = Ks + kPiece * d;
  float* Es = Vs + kPiece * d;   // errors; for LN first y = K W_a
  float* Xs = Es + kPiece * d;   // LN: read-out pre-activations
  float* Ss = Xs + kPiece * d;   // [16][16]
  float* vec = Ss + kPiece * kPiece;  // [4][64]: beta_r, beta_a (bias); gamma, beta (LN)
  float* tok = vec + 4 * 64;     // [2][16]: per-token rate (or row scales), spare

  const int unit = blockIdx.x;
  const int h = unit % p.H;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const float eta = kVar == kVarTokenEta ? 0.f : p.rate[h];  // per-token rates come from tok_rate
  const float mbeta = kVar == kVarMomentum ? p.mbeta[h] : 0.f;
  const size_t base = static_cast<size_t>(unit) * p.T * d;
  const T* Q = static_cast<const T*>(p.Q) + base;
  const T* K = static_cast<const T*>(p.K) + base;
  const T* V = static_cast<const T*>(p.V) + base;
  T* Z = static_cast<T*>(p.Z) + base;

  const float* W0 = p.W0 + static_cast<size_t>(h) * d * d;
  for (int x = tid; x < d * d; x += kThreads) {
    Wr[x] = Wa[x] = W0[x];
    if (kVar == kVarMomentum) Mr[x] = 0.f;
  }
  if (kVar == kVarBias)
    for (int j = tid; j < d; j += kThreads) vec[j] = vec[64 + j] = p.vec0[static_cast<size_t>(h) * d + j];
  if (kVar == kVarLn)
    for (int j = tid; j < d; j += kThreads) {
      vec[j] = p.vec0[static_cast<size_t>(h) * d + j];       // gamma
      vec[64 + j] = p.vec1[static_cast<size_t>(h) * d + j];  // beta
    }
  __syncthreads();

  for (int t0 = 0; t0 < p.T;) {
    const int chunk_end = min((t0 / p.b + 1) * p.b, p.T);
    const int t1 = min(t0 + kPiece, chunk_end);
    const int n = t1 - t0;
    for (int x = tid; x < n * d; x += kThreads) {
      const size_t g = static_cast<size_t>(t0) * d + x;
      Qs[x] = ld_in<T>(Q + g);
      Ks[x] = ld_in<T>(K + g);
      Vs[x] = ld_in<T>(V + g);
    }
    if (kVar == kVarTokenEta && tid < n) tok[tid] = p.tok_rate[static_cast<size_t>(unit) * p.T + t0 + tid];
    __syncthreads();

    // E from the chunk-start state (LN: y = K W_a first).
    for (int x = tid; x < n * d; x += kThreads) {
      const int t = x / d, j = x % d;
      float s = 0.f;
      for (int i = 0; i < d; ++i) s = fmaf(Ks[t * d + i], Wa[i * d + j], s);
      if (kVar == kVarLn)
        Es[x] = s;
      else if (kVar == kVarBias)
        Es[x] = s + vec[64 + j] - Vs[x];
      else
        Es[x] = s - Vs[x];
    }
    // Intra-piece read-out weights S[t][i], i <= t.
    for (int x = tid; x < n * n; x += kThreads) {
      const int t = x / n, i = x % n;
      float s = 0.f;
      if (i <= t) {
        for (int k = 0; k < d; ++k) s = fmaf(Qs[t * d + k], Ks[i * d + k], s);
        if (kVar == kVarBias) s += 1.f;
        if (kVar == kVarTokenEta) s *= tok[i];
        if (kVar == kVarMomentum) s *= 1.f - powf(mbeta, static_cast<float>(t - i + 1));
      }
      Ss[t * kPiece + i] = s;
    }
    __syncthreads();
    if (kVar == kVarLn) {
      // e = (g - mean(g) - x mean(g x)) / s with x the normalised y, g = gamma (k + gamma x + beta - v)
      normalise_rows(Es, tok + kPiece, n, d, warp, lane);
      __syncwarp();
      for (int t = warp; t < n; t += kWarpsV) {
        float sg = 0.f, sgx = 0.f;
        for (int j = lane; j < d; j += 32) {
          const float x = Es[t * d + j];
          const float gj = vec[j] * (Ks[t * d + j] + vec[j] * x + vec[64 + j] - Vs[t * d + j]);
          sg += gj;
          sgx += gj * x;
        }
        const float mg = warp_sum(sg) / d, mgx = warp_sum(sgx) / d;
        const float inv = tok[kPiece + t];
        for (int j = lane; j < d; j += 32) {
          const float x = Es[t * d + j];
          const float gj = vec[j] * (Ks[t * d + j] + vec[j] * x + vec[64 + j] - Vs[t * d + j]);
          Es[t * d + j] = (gj - mg - x * mgx) * inv;
        }
      }
      __syncthreads();
    }

    // Read-out with the running state at the piece start, plus the piece's own terms.
    for (int x = tid; x < n * d; x += kThreads) {
      const int t = x / d, j = x % d;
      float qw = 0.f, se = 0.f, qm = 0.f;
      for (int i = 0; i < d; ++i) qw = fmaf(Qs[t * d + i], Wr[i * d + j], qw);
      for (int i = 0; i <= t; ++i) se = fmaf(Ss[t * kPiece + i], Es[i * d + j], se);
      float out;
      if (kVar == kVarMomentum) {
        for (int i = 0; i < d; ++i) qm = fmaf(Qs[t * d + i], Mr[i * d + j], qm);
        // c_{t+1} = beta + ... + beta^(t+1)
        float c = 0.f, pw = 1.f;
        for (int k = 0; k <= t; ++k) {
          pw *= mbeta;
          c += pw;
        }
        out = qw - eta * c * qm - eta * se;
      } else if (kVar == kVarTokenEta) {
        out = qw - se;
      } else if (kVar == kVarBias) {
        out = qw + vec[j] - eta * se;
      } else {
        out = qw - eta * se;
      }
      if (kVar == kVarLn)
        Xs[x] = out;
      else
        st_out<T>(Z + static_cast<size_t>(t0) * d + x, out);
    }
    __syncthreads();
    if (kVar == kVarLn) {
      normalise_rows(Xs, tok + kPiece, n, d, warp, lane);
      __syncthreads();
      for (int x = tid; x < n * d; x += kThreads) {
        const int j = x % d;
        st_out<T>(Z + static_cast<size_t>(t0) * d + x, Qs[x] + vec[j] * Xs[x] + vec[64 + j]);
      }
    }

    // State update by the piece's gradients.
    if (kVar == kVarMomentum) {
      float cn = 0.f, pw = 1.f;
      for (int k = 0; k < n; ++k) {
        pw *= mbeta;
        cn += pw;
      }
      const float bn = pw;  // beta^n
      for (int x = tid; x < d * d; x += kThreads) {
        const int i = x / d, j = x % d;
        float kd = 0.f, kw = 0.f, wk = 1.f;  // wk = beta^(n-1-t), walking t downwards
        for (int t = n - 1; t >= 0; --t) {
          const float ke = Ks[t * d + i] * Es[t * d + j];
          kw = fmaf(wk, ke, kw);
          kd = fmaf(1.f - wk * mbeta, ke, kd);  // 1 - beta^(n-t)
          wk *= mbeta;
        }
        const float m = Mr[x];
        Wr[x] -= eta * (cn * m + kd);
        Mr[x] = bn * m + (1.f - mbeta) * kw;
      }
    } else {
      for (int x = tid; x < d * d; x += kThreads) {
        const int i = x / d, j = x % d;
        float s = 0.f;
        for (int t = 0; t < n; ++t) {
          const float ke = Ks[t * d + i] * Es[t * d + j];
          s = kVar == kVarTokenEta ? fmaf(tok[t], ke, s) : s + ke;
        }
        Wr[x] -= (kVar == kVarTokenEta ? 1.f : eta) * s;
      }
      if (kVar == kVarBias && tid < d) {
        float s = 0.f;
        for (int t = 0; t < n; ++t) s += Es[t * d + tid];
        vec[tid] -= eta * s;
      }
    }
    __syncthreads();
    if (t1 == chunk_end) {
      for (int x = tid; x < d * d; x += kThreads) Wa[x] = Wr[x];
      if (kVar == kVarBias && tid < d) vec[64 + tid] = vec[tid];
      __syncthreads();
    }
    t0 = t1;
  }
  float* Wo = p.W_out + static_cast<size_t>(unit) * d * d;
  for (int x = tid; x < d * d; x += kThreads) Wo[x] = Wr[x];
  if (kVar == kVarMomentum) {
    float* Mo = p.aux_out + static_cast<size_t>(unit) * d * d;
    for (int x = tid; x < d * d; x += kThreads) Mo[x] = Mr[x];
  }
  if (kVar == kVarBias) {
    float* bo = p.aux_out + static_cast<size_t>(unit) * d;
    for (int j = tid; j < d; j += kThreads) bo[j] = vec[j];
  }
}

template <int kVar>
cudaError_t launch_typed(const VariantParams& p, cudaStream_t stream) {
  const size_t floats = (kVar == kVarMomentum ? 3 : 2) * static_cast<size_t>(p.d) * p.d + 6 * kPiece * p.d +
                        kPiece * kPiece + 4 * 64 + 2 * kPiece;
  const size_t smem = floats * sizeof(float);
  cudaError_t err;
  if (p.bf16) {
    err = cudaFuncSetAttribute(linear_variant_kernel<__nv_bfloat16, kVar>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    linear_variant_kernel<__nv_bfloat16, kVar><<<p.units, kThreads, smem, stream>>>(p);
  } else {
    err = cudaFuncSetAttribute(linear_variant_kernel<float, kVar>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    linear_variant_kernel<float, kVar><<<p.units, kThreads, smem, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_linear_variant(const VariantParams& p, cudaStream_t stream) {
  if (p.units == 0) return cudaSuccess;
  switch (p.variant) {
    case kVarBias: return launch_typed<kVarBias>(p, stream);
    case kVarTokenEta: return launch_typed<kVarTokenEta>(p, stream);
    case kVarLn: return launch_typed<kVarLn>(p, stream);
    case kVarMomentum: return launch_typed<kVarMomentum>(p, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace ttt
