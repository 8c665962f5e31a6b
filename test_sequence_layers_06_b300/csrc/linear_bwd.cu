// Backward of the chunked TTT-Linear scan in fp32 arithmetic: fp32 or bf16
// operands (dQ, dK, dV in the operands' dtype), d <= 64, b <= 64.
//
// The outer loop trains W0 and the projections that make Q, K, V by
// backpropagating through the inner loop ("5 · TestingTime 训练与长上下文",
// section 2.2). For upstream gradients dZ and dW_out this computes dQ, dK, dV,
// d eta and dW0 of the chunk rule of section 1.1 (gradients of the whole chunk
// at the chunk-start weights, read-out with the updated weights):
//   E = K_c W - V_c,  S = tril(Q_c K_c^T),  Z_c = Q_c W - eta S E,  W' = W - eta K_c^T E.
// Reversed chunk by chunk from G = dW_out (G: gradient of the next chunk's
// start state), with P = -eta tril(dZ_c E^T) the gradient of S:
//   dE   = -eta K_c G - eta S^T dZ_c
//   dQ_c = dZ_c W^T + P K_c
//   dK_c = -eta E G^T + P^T Q_c + dE W^T
//   dV_c = -dE
//   d eta += -sum(E * (K_c G)) - sum(S * (dZ_c E^T))
//   G   <- G + Q_c^T dZ_c + K_c^T dE
// and dW0 = G after the first chunk. W0 and eta are shared by the batch rows,
// so their gradients are summed over rows by a second kernel.
//
// Design: one CTA per (batch row, head). A forward pass keeps every
// chunk-start state in the workspace; the backward pass reloads them in
// reverse. Every matrix of a chunk sits in shared memory and every product is
// a plain fp32 loop spread over the CTA's threads: the general form, for the
// 1e-4 bar of fp32 operands and the shapes linear_bwd_mma.cu does not take.
#include "ttt_device.cuh"
#include "kernels.h"

namespace ttt {
namespace {

constexpr int kBwdThreads = 256;

template <typename T>
__device__ __forceinline__ float ldv(const void* p, size_t i) {
  return static_cast<float>(static_cast<const T*>(p)[i]);
}
template <typename T>
__device__ __forceinline__ void stv(void* p, size_t i, float v) {
  static_cast<T*>(p)[i] = static_cast<T>(v);
}

template <typename Tin>
__global__ void __launch_bounds__(kBwdThreads) linear_bwd_kernel(LinearBwdParams p) {
  extern __shared__ __align__(16) float bsm[];
  const int d = p.d, b = p.b, T = p.T;
  const int unit = blockIdx.x;
  const int h = unit % p.H;
  const int tid = threadIdx.x;
  const float eta = p.eta[h];
  const int nch = (T + b - 1) / b;
  float* W = bsm;            // [d][d]   chunk-start state
  float* G = W + d * d;      // [d][d]   gradient of the next chunk's start state
  float* Qc = G + d * d;     // [b][d]
  float* Kc = Qc + b * d;
  float* Vc = Kc + b * d;
  float* dZc = Vc + b * d;
  float* E = dZc + b * d;
  float* dE = E + b * d;
  float* KG = dE + b * d;    // K_c G
  float* S = KG + b * d;     // [b][b]  tril(Q_c K_c^T)
  float* P = S + b * b;      // [b][b]  -eta tril(dZ_c E^T)
  float* red = P + b * b;    // [kBwdThreads]
  const size_t base = static_cast<size_t>(unit) * T * d;
  float* states = p.states + static_cast<size_t>(unit) * nch * d * d;

  // ---------------------------------------------------------------- forward: chunk-start states
  for (int i = tid; i < d * d; i += kBwdThreads) W[i] = p.W0[static_cast<size_t>(h) * d * d + i];
  __syncthreads();
  for (int c = 0; c < nch; ++c) {
    const int c0 = c * b, n = min(b, T - c0);
    for (int i = tid; i < d * d; i += kBwdThreads) states[static_cast<size_t>(c) * d * d + i] = W[i];
    for (int x = tid; x < n * d; x += kBwdThreads) {
      Kc[x] = ldv<Tin>(p.K, base + static_cast<size_t>(c0) * d + x);
      Vc[x] = ldv<Tin>(p.V, base + static_cast<size_t>(c0) * d + x);
    }
    __syncthreads();
    for (int x = tid; x < n * d; x += kBwdThreads) {  // E = K_c W - V_c
      const int t = x / d, j = x % d;
      float acc = -Vc[x];
      for (int k = 0; k < d; ++k) acc = fmaf(Kc[t * d + k], W[k * d + j], acc);
      E[x] = acc;
    }
    __syncthreads();
    for (int x = tid; x < d * d; x += kBwdThreads) {  // W -= eta K_c^T E
      const int i = x / d, j = x % d;
      float acc = 0.f;
      for (int t = 0; t < n; ++t) acc = fmaf(Kc[t * d + i], E[t * d + j], acc);
      W[x] -= eta * acc;
    }
    __syncthreads();
  }

  // ---------------------------------------------------------------- backward, last chunk first
  for (int i = tid; i < d * d; i += kBwdThreads) G[i] = p.dW_out[static_cast<size_t>(unit) * d * d + i];
  float deta = 0.f;
  __syncthreads();
  for (int c = nch - 1; c >= 0; --c) {
    const int c0 = c * b, n = min(b, T - c0);
    const size_t off = base + static_cast<size_t>(c0) * d;
    for (int i = tid; i < d * d; i += kBwdThreads) W[i] = states[static_cast<size_t>(c) * d * d + i];
    for (int x = tid; x < n * d; x += kBwdThreads) {
      Qc[x] = ldv<Tin>(p.Q, off + x);
      Kc[x] = ldv<Tin>(p.K, off + x);
      Vc[x] = ldv<Tin>(p.V, off + x);
      dZc[x] = ldv<Tin>(p.dZ, off + x);
    }
    __syncthreads();
    for (int x = tid; x < n * d; x += kBwdThreads) {  // E = K_c W - V_c, KG = K_c G
      const int t = x / d, j = x % d;
      float e = -Vc[x], kg = 0.f;
      for (int k = 0; k < d; ++k) {
        e = fmaf(Kc[t * d + k], W[k * d + j], e);
        kg = fmaf(Kc[t * d + k], G[k * d + j], kg);
      }
      E[x] = e;
      KG[x] = kg;
    }
    for (int x = tid; x < n * n; x += kBwdThreads) {  // S = tril(Q_c K_c^T), diagonal kept
      const int t = x / n, t2 = x % n;
      float acc = 0.f;
      if (t2 <= t)
        for (int i = 0; i < d; ++i) acc = fmaf(Qc[t * d + i], Kc[t2 * d + i], acc);
      S[x] = acc;
    }
    __syncthreads();
    for (int x = tid; x < n * n; x += kBwdThreads) {  // P = -eta tril(dZ_c E^T); d eta from S E
      const int t = x / n, t2 = x % n;
      float pv = 0.f;
      if (t2 <= t) {
        for (int j = 0; j < d; ++j) pv = fmaf(dZc[t * d + j], E[t2 * d + j], pv);
        deta -= S[x] * pv;
      }
      P[x] = -eta * pv;
    }
    for (int x = tid; x < n * d; x += kBwdThreads) {  // dE = -eta K_c G - eta S^T dZ_c; d eta from K^T E
      const int t = x / d, j = x % d;
      deta -= E[x] * KG[x];
      float acc = 0.f;
      for (int t2 = t; t2 < n; ++t2) acc = fmaf(S[t2 * n + t], dZc[t2 * d + j], acc);
      dE[x] = -eta * (KG[x] + acc);
    }
    __syncthreads();
    for (int x = tid; x < n * d; x += kBwdThreads) {  // dQ_c, dK_c, dV_c
      const int t = x / d, i = x % d;
      float aq = 0.f, ak = 0.f, eg = 0.f;
      for (int j = 0; j < d; ++j) {
        aq = fmaf(dZc[t * d + j], W[i * d + j], aq);
        ak = fmaf(dE[t * d + j], W[i * d + j], ak);
        eg = fmaf(E[t * d + j], G[i * d + j], eg);
      }
      for (int t2 = 0; t2 <= t; ++t2) aq = fmaf(P[t * n + t2], Kc[t2 * d + i], aq);
      for (int t2 = t; t2 < n; ++t2) ak = fmaf(P[t2 * n + t], Qc[t2 * d + i], ak);
      stv<Tin>(p.dQ, off + x, aq);
      stv<Tin>(p.dK, off + x, ak - eta * eg);
      stv<Tin>(p.dV, off + x, -dE[x]);
    }
    __syncthreads();  // G is read above; update it only now
    for (int x = tid; x < d * d; x += kBwdThreads) {  // G += Q_c^T dZ_c + K_c^T dE
      const int i = x / d, j = x % d;
      float acc = 0.f;
      for (int t = 0; t < n; ++t) acc = fmaf(Qc[t * d + i], dZc[t * d + j], fmaf(Kc[t * d + i], dE[t * d + j], acc));
      G[x] += acc;
    }
    __syncthreads();
  }

  // ---------------------------------------------------------------- per-unit partials of dW0, d eta
  float* part = p.partial + static_cast<size_t>(unit) * (d * d + 1);
  for (int i = tid; i < d * d; i += kBwdThreads) part[i] = G[i];
  red[tid] = deta;
  __syncthreads();
  for (int s = kBwdThreads / 2; s > 0; s >>= 1) {
    if (tid < s) red[tid] += red[tid + s];
    __syncthreads();
  }
  if (tid == 0) part[d * d] = red[0];
}

// dW0[h] and d eta[h]: sums over the batch rows of the per-unit partials.
__global__ void __launch_bounds__(kBwdThreads) linear_bwd_reduce_kernel(LinearBwdParams p) {
  const int h = blockIdx.x;
  const int d = p.d;
  for (int i = threadIdx.x; i <= d * d; i += kBwdThreads) {
    float acc = 0.f;
    for (int n = 0; n < p.B; ++n) acc += p.partial[static_cast<size_t>(n * p.H + h) * (d * d + 1) + i];
    if (i < d * d)
      p.dW0[static_cast<size_t>(h) * d * d + i] = acc;
    else
      p.deta[h] = acc;
  }
}

}  // namespace

size_t linear_bwd_smem_bytes(int d, int b) {
  return (static_cast<size_t>(2) * d * d + static_cast<size_t>(7) * b * d + static_cast<size_t>(2) * b * b +
          kBwdThreads) *
         sizeof(float);
}

bool linear_bwd_supported(int d, int b) {
  return d >= 1 && d <= 64 && b >= 1 && b <= 64 && linear_bwd_smem_bytes(d, b) <= 227 * 1024;
}

size_t linear_bwd_scratch_bytes(int units, int T, int d, int b) {
  const size_t nch = (static_cast<size_t>(T) + b - 1) / b;
  return static_cast<size_t>(units) * nch * d * d * sizeof(float) +
         static_cast<size_t>(units) * (static_cast<size_t>(d) * d + 1) * sizeof(float);
}

cudaError_t launch_linear_bwd(const LinearBwdParams& p, cudaStream_t stream) {
  const size_t smem = linear_bwd_smem_bytes(p.d, p.b);
  auto kern = p.bf16 ? linear_bwd_kernel<__nv_bfloat16> : linear_bwd_kernel<float>;
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  kern<<<p.units, kBwdThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_linear_bwd_reduce(const LinearBwdParams& p, cudaStream_t stream) {
  linear_bwd_reduce_kernel<<<p.H, kBwdThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace ttt
