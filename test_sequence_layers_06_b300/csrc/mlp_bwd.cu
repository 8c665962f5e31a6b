// Backward of the chunked TTT-MLP scan in fp32 arithmetic (fp32 or bf16
// operands), d <= 64, hidden m = 4d, any chunk size: the vector-Jacobian product
// of (Z, W1_out, W2_out) with respect to (Q, K, V, eta, W1_0, W2_0).
//
// The forward it reverses ("Test-Time Training (TTT) guide", section 3: two
// layers, hidden 4x, GELU; "5 · TestingTime 训练与长上下文", section 1.1: the
// gradients of a chunk at its start weights, read out in the dual form), per
// chunk with start weights P1 [d][m], P2 [m][d]:
//   U = K P1, A = s(U), G = A P2 - V, D1 = G P2^T, D = D1 .* s'(U)
//   S = tril(Q K^T), Hq = Q P1 - eta S D, Aq = s(Hq), R = tril(Aq A^T)
//   Z = Aq P2 - eta R G,   P1' = P1 - eta K^T D,   P2' = P2 - eta A^T G
// with s the tanh-GELU of Hendrycks and Gimpel (2016). The backward walks the
// chunks last first from the gradients G1, G2 of the next chunk's start weights
// (dW1_out, dW2_out at the end) and applies the chain rule to each line above in
// reverse order; s'' enters through D's dependence on U. The outer loop trains
// W1_0, W2_0 and eta through this ("5 · TestingTime 训练与长上下文", section 2.2).
//
// Design: a parity form. One CTA of 256 threads per (batch row, head); a forward
// pass keeps every chunk-start (P1, P2) in the workspace, and every matrix of a
// chunk lives in the workspace too (fp32), read back through L1/L2. Each product
// is a plain loop over the CTA's threads followed by a CTA barrier (global
// writes are visible to the whole CTA after __syncthreads).
#include "ttt_device.cuh"
#include "kernels.h"

namespace ttt {
namespace {

constexpr int kThreads = 256;
constexpr float kGeluC = 0.7978845608028654f;  // sqrt(2 / pi)
constexpr float kGeluA = 0.044715f;

template <typename T>
__device__ __forceinline__ float ldv(const void* p, size_t i) {
  return static_cast<float>(static_cast<const T*>(p)[i]);
}
template <typename T>
__device__ __forceinline__ void stv(void* p, size_t i, float v) {
  static_cast<T*>(p)[i] = static_cast<T>(v);
}

// s, s' and s'' of the tanh-GELU at u.
__device__ __forceinline__ void gelu3(float u, float* s, float* s1, float* s2) {
  const float k = kGeluC * (1.f + 3.f * kGeluA * u * u);
  const float th = tanhf(kGeluC * (u + kGeluA * u * u * u));
  const float th1 = (1.f - th * th) * k;
  const float th2 = -2.f * th * th1 * k + (1.f - th * th) * 6.f * kGeluA * kGeluC * u;
  if (s) *s = 0.5f * u * (1.f + th);
  if (s1) *s1 = 0.5f * (1.f + th) + 0.5f * u * th1;
  if (s2) *s2 = th1 + 0.5f * u * th2;
}

// C = alpha * opA(A) opB(B) (+ C when acc), C [M][N] with row stride ldc.
// opA(A)[i][k] = TA ? A[k][i] : A[i][k] (row stride lda), likewise opB. With
// tril only entries j <= i are formed (the rest are written 0 unless acc).
// Ends with a CTA barrier.
template <bool TA, bool TB>
__device__ void mm(float* C, int ldc, const float* A, int lda, const float* B, int ldb, int M, int N, int K,
                   float alpha, bool acc, bool tril) {
  for (int x = threadIdx.x; x < M * N; x += kThreads) {
    const int i = x / N, j = x % N;
    float s = 0.f;
    if (!tril || j <= i)
      for (int k = 0; k < K; ++k) s = fmaf(TA ? A[k * lda + i] : A[i * lda + k], TB ? B[j * ldb + k] : B[k * ldb + j], s);
    float* c = C + i * ldc + j;
    *c = acc ? *c + alpha * s : alpha * s;
  }
  __syncthreads();
}

__device__ float block_sum(float v, float* red) {
  red[threadIdx.x] = v;
  __syncthreads();
  for (int s = kThreads / 2; s > 0; s >>= 1) {
    if (threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
    __syncthreads();
  }
  const float r = red[0];
  __syncthreads();
  return r;
}

template <typename Tin>
__global__ void __launch_bounds__(kThreads) mlp_bwd_kernel(MlpBwdParams p) {
  __shared__ float red[kThreads];
  const int d = p.d, m = p.m, b = p.b, T = p.T;
  const int unit = blockIdx.x, h = unit % p.H, tid = threadIdx.x;
  const float e = p.eta[h];
  const int nch = (T + b - 1) / b;
  const int cap = min(b, T);
  const size_t dm = static_cast<size_t>(d) * m;
  const size_t base = static_cast<size_t>(unit) * T * d;
  // workspace of this unit
  float* ws = p.scratch + static_cast<size_t>(unit) * mlp_bwd_unit_floats(T, d, b);
  float* states = ws;                                 // [nch][P1 d*m | P2 m*d]
  float* G1 = states + static_cast<size_t>(nch) * 2 * dm;
  float* G2 = G1 + dm;
  float* dP1 = G2 + dm;
  float* dP2 = dP1 + dm;
  float* Qc = dP2 + dm;                              // [cap][d] each
  float* Kc = Qc + cap * d;
  float* Vc = Kc + cap * d;
  float* dZc = Vc + cap * d;
  float* Gm = dZc + cap * d;
  float* dG = Gm + cap * d;
  float* dKc = dG + cap * d;
  float* dQc = dKc + cap * d;
  float* A = dQc + cap * d;                          // [cap][m] each
  float* S1 = A + cap * m;
  float* S2 = S1 + cap * m;
  float* D1 = S2 + cap * m;
  float* Dm = D1 + cap * m;
  float* Aq = Dm + cap * m;
  float* Sq1 = Aq + cap * m;
  float* dA = Sq1 + cap * m;
  float* dD = dA + cap * m;
  float* dAq = dD + cap * m;
  float* dU = dAq + cap * m;
  float* Sm = dU + cap * m;                          // [cap][cap] each
  float* Rm = Sm + cap * cap;
  float* Tm = Rm + cap * cap;

  auto load_chunk = [&](size_t off, int n, bool all) {
    for (int x = tid; x < n * d; x += kThreads) {
      Kc[x] = ldv<Tin>(p.K, off + x);
      Vc[x] = ldv<Tin>(p.V, off + x);
      if (all) {
        Qc[x] = ldv<Tin>(p.Q, off + x);
        dZc[x] = ldv<Tin>(p.dZ, off + x);
      }
    }
    __syncthreads();
  };
  // U = Kc P1 -> A = s(U), S1 = s'(U), S2 = s''(U) (U itself is kept in S2's place first)
  auto gelu_of_keys = [&](const float* P1, int n, bool second) {
    mm<false, false>(S2, m, Kc, d, P1, m, n, m, d, 1.f, false, false);
    for (int x = tid; x < n * m; x += kThreads) {
      float s, s1, s2;
      gelu3(S2[x], &s, &s1, second ? &s2 : nullptr);
      A[x] = s;
      S1[x] = s1;
      S2[x] = second ? s2 : 0.f;
    }
    __syncthreads();
  };

  // ---------------------------------------------------------------- forward: chunk-start weights
  for (size_t x = tid; x < dm; x += kThreads) {
    states[x] = p.W1_0[static_cast<size_t>(h) * dm + x];
    states[dm + x] = p.W2_0[static_cast<size_t>(h) * dm + x];
  }
  __syncthreads();
  for (int c = 0; c + 1 < nch; ++c) {
    const int c0 = c * b, n = min(b, T - c0);
    const float* P1 = states + static_cast<size_t>(c) * 2 * dm;
    const float* P2 = P1 + dm;
    float* N1 = states + static_cast<size_t>(c + 1) * 2 * dm;
    float* N2 = N1 + dm;
    load_chunk(base + static_cast<size_t>(c0) * d, n, false);
    gelu_of_keys(P1, n, false);
    mm<false, false>(Gm, d, A, m, P2, d, n, d, m, 1.f, false, false);           // G = A P2 - V
    for (int x = tid; x < n * d; x += kThreads) Gm[x] -= Vc[x];
    __syncthreads();
    mm<false, true>(Dm, m, Gm, d, P2, d, n, m, d, 1.f, false, false);           // D = (G P2^T) .* s'(U)
    for (int x = tid; x < n * m; x += kThreads) Dm[x] *= S1[x];
    for (size_t x = tid; x < dm; x += kThreads) {
      N1[x] = P1[x];
      N2[x] = P2[x];
    }
    __syncthreads();
    mm<true, false>(N1, m, Kc, d, Dm, m, d, m, n, -e, true, false);             // P1 - eta K^T D
    mm<true, false>(N2, d, A, m, Gm, d, m, d, n, -e, true, false);              // P2 - eta A^T G
  }

  // ---------------------------------------------------------------- backward, last chunk first
  for (size_t x = tid; x < dm; x += kThreads) {
    G1[x] = p.dW1_out[static_cast<size_t>(unit) * dm + x];
    G2[x] = p.dW2_out[static_cast<size_t>(unit) * dm + x];
  }
  float deta = 0.f;
  __syncthreads();
  for (int c = nch - 1; c >= 0; --c) {
    const int c0 = c * b, n = min(b, T - c0);
    const size_t off = base + static_cast<size_t>(c0) * d;
    const float* P1 = states + static_cast<size_t>(c) * 2 * dm;
    const float* P2 = P1 + dm;
    load_chunk(off, n, true);
    // the chunk's forward
    gelu_of_keys(P1, n, true);
    mm<false, false>(Gm, d, A, m, P2, d, n, d, m, 1.f, false, false);
    for (int x = tid; x < n * d; x += kThreads) Gm[x] -= Vc[x];
    __syncthreads();
    mm<false, true>(D1, m, Gm, d, P2, d, n, m, d, 1.f, false, false);           // D1 = G P2^T
    for (int x = tid; x < n * m; x += kThreads) Dm[x] = D1[x] * S1[x];
    __syncthreads();
    mm<false, true>(Sm, cap, Qc, d, Kc, d, n, n, d, 1.f, false, true);          // S = tril(Q K^T)
    mm<false, false>(Aq, m, Qc, d, P1, m, n, m, d, 1.f, false, false);          // Hq = Q P1 - eta S D
    mm<false, false>(Aq, m, Sm, cap, Dm, m, n, m, n, -e, true, false);
    for (int x = tid; x < n * m; x += kThreads) gelu3(Aq[x], &Aq[x], &Sq1[x], nullptr);
    __syncthreads();
    mm<false, true>(Rm, cap, Aq, m, A, m, n, n, m, 1.f, false, true);           // R = tril(Aq A^T)

    // P1' = P1 - eta K^T D,  P2' = P2 - eta A^T G
    for (size_t x = tid; x < dm; x += kThreads) {
      dP1[x] = G1[x];
      dP2[x] = G2[x];
    }
    mm<false, true>(dKc, d, Dm, m, G1, m, n, d, m, -e, false, false);           // dK = -eta D G1^T
    mm<false, false>(dD, m, Kc, d, G1, m, n, m, d, 1.f, false, false);          // K G1
    mm<false, true>(dA, m, Gm, d, G2, d, n, m, d, 1.f, false, false);           // G G2^T
    float part = 0.f;
    for (int x = tid; x < n * m; x += kThreads) {  // d eta -= sum (K^T D) .* G1 + sum (A^T G) .* G2
      part += Dm[x] * dD[x] + A[x] * dA[x];
      dD[x] *= -e;
      dA[x] *= -e;
    }
    deta -= part;
    __syncthreads();
    mm<false, false>(dG, d, A, m, G2, d, n, d, m, -e, false, false);            // dG = -eta A G2
    // Z = Aq P2 - eta R G
    mm<false, true>(dAq, m, dZc, d, P2, d, n, m, d, 1.f, false, false);         // dAq = dZ P2^T
    mm<true, false>(dP2, d, Aq, m, dZc, d, m, d, n, 1.f, true, false);          // dP2 += Aq^T dZ
    mm<false, true>(Tm, cap, dZc, d, Gm, d, n, n, d, 1.f, false, true);         // tril(dZ G^T)
    part = 0.f;
    for (int x = tid; x < n * n; x += kThreads) {  // d eta -= sum (R G) .* dZ;  dR = -eta tril(dZ G^T)
      const int i = x / n, j = x % n;
      part += Rm[i * cap + j] * Tm[i * cap + j];
    }
    deta -= part;
    __syncthreads();
    for (int x = tid; x < n * n; x += kThreads) Tm[(x / n) * cap + x % n] *= -e;
    __syncthreads();
    mm<true, false>(dG, d, Rm, cap, dZc, d, n, d, n, -e, true, false);          // dG -= eta R^T dZ
    // R = tril(Aq A^T)
    mm<false, false>(dAq, m, Tm, cap, A, m, n, m, n, 1.f, true, false);         // dAq += dR A
    mm<true, false>(dA, m, Tm, cap, Aq, m, n, m, n, 1.f, true, false);          // dA += dR^T Aq
    // Aq = s(Hq): dHq in dAq's place
    for (int x = tid; x < n * m; x += kThreads) dAq[x] *= Sq1[x];
    __syncthreads();
    // Hq = Q P1 - eta S D
    mm<false, true>(dQc, d, dAq, m, P1, m, n, d, m, 1.f, false, false);         // dQ = dHq P1^T
    mm<true, false>(dP1, m, Qc, d, dAq, m, d, m, n, 1.f, true, false);          // dP1 += Q^T dHq
    mm<false, true>(Tm, cap, dAq, m, Dm, m, n, n, m, 1.f, false, true);         // tril(dHq D^T)
    part = 0.f;
    for (int x = tid; x < n * n; x += kThreads) {  // d eta -= sum (S D) .* dHq;  dS = -eta tril(dHq D^T)
      const int i = x / n, j = x % n;
      part += Sm[i * cap + j] * Tm[i * cap + j];
    }
    deta -= part;
    __syncthreads();
    for (int x = tid; x < n * n; x += kThreads) Tm[(x / n) * cap + x % n] *= -e;
    __syncthreads();
    mm<true, false>(dD, m, Sm, cap, dAq, m, n, m, n, -e, true, false);          // dD -= eta S^T dHq
    // S = tril(Q K^T)
    mm<false, false>(dQc, d, Tm, cap, Kc, d, n, d, n, 1.f, true, false);        // dQ += dS K
    mm<true, false>(dKc, d, Tm, cap, Qc, d, n, d, n, 1.f, true, false);         // dK += dS^T Q
    // D = D1 .* s'(U), D1 = G P2^T:  dD1 in dD's place, dU = dD .* D1 .* s''(U)
    for (int x = tid; x < n * m; x += kThreads) {
      dU[x] = dD[x] * D1[x] * S2[x];
      dD[x] *= S1[x];
    }
    __syncthreads();
    mm<false, false>(dG, d, dD, m, P2, d, n, d, m, 1.f, true, false);           // dG += dD1 P2
    mm<true, false>(dP2, d, dD, m, Gm, d, m, d, n, 1.f, true, false);           // dP2 += dD1^T G
    // G = A P2 - V
    for (int x = tid; x < n * d; x += kThreads) stv<Tin>(p.dV, off + x, -dG[x]);
    mm<false, true>(dA, m, dG, d, P2, d, n, m, d, 1.f, true, false);            // dA += dG P2^T
    mm<true, false>(dP2, d, A, m, dG, d, m, d, n, 1.f, true, false);            // dP2 += A^T dG
    // A = s(U), U = K P1
    for (int x = tid; x < n * m; x += kThreads) dU[x] += dA[x] * S1[x];
    __syncthreads();
    mm<false, true>(dKc, d, dU, m, P1, m, n, d, m, 1.f, true, false);           // dK += dU P1^T
    mm<true, false>(dP1, m, Kc, d, dU, m, d, m, n, 1.f, true, false);           // dP1 += K^T dU
    for (int x = tid; x < n * d; x += kThreads) {
      stv<Tin>(p.dQ, off + x, dQc[x]);
      stv<Tin>(p.dK, off + x, dKc[x]);
    }
    for (size_t x = tid; x < dm; x += kThreads) {
      G1[x] = dP1[x];
      G2[x] = dP2[x];
    }
    __syncthreads();
  }

  // ---------------------------------------------------------------- per-unit partials of dW1, dW2, d eta
  float* part = p.partial + static_cast<size_t>(unit) * (2 * dm + 1);
  for (size_t x = tid; x < dm; x += kThreads) {
    part[x] = G1[x];
    part[dm + x] = G2[x];
  }
  const float total = block_sum(deta, red);
  if (tid == 0) part[2 * dm] = total;
}

// dW1[h], dW2[h], d eta[h]: sums over the batch rows of the per-unit partials.
__global__ void __launch_bounds__(kThreads) mlp_bwd_reduce_kernel(MlpBwdParams p) {
  const int h = blockIdx.x;
  const size_t dm = static_cast<size_t>(p.d) * p.m;
  for (size_t i = threadIdx.x; i <= 2 * dm; i += kThreads) {
    float acc = 0.f;
    for (int n = 0; n < p.B; ++n) acc += p.partial[static_cast<size_t>(n * p.H + h) * (2 * dm + 1) + i];
    if (i < dm)
      p.dW1[static_cast<size_t>(h) * dm + i] = acc;
    else if (i < 2 * dm)
      p.dW2[static_cast<size_t>(h) * dm + i - dm] = acc;
    else
      p.deta[h] = acc;
  }
}

}  // namespace

size_t mlp_bwd_scratch_bytes(int units, int T, int d, int b) {
  const size_t dm = static_cast<size_t>(d) * 4 * d;
  return (static_cast<size_t>(units) * mlp_bwd_unit_floats(T, d, b) + static_cast<size_t>(units) * (2 * dm + 1)) *
         sizeof(float);
}

cudaError_t launch_mlp_bwd(const MlpBwdParams& p, cudaStream_t stream) {
  if (p.bf16)
    mlp_bwd_kernel<__nv_bfloat16><<<p.units, kThreads, 0, stream>>>(p);
  else
    mlp_bwd_kernel<float><<<p.units, kThreads, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  mlp_bwd_reduce_kernel<<<p.H, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace ttt
