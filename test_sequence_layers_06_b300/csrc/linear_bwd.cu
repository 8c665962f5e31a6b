// Backward of the chunked TTT-Linear scan in fp32 arithmetic: fp32 or bf16
// operands (dQ, dK, dV in the operands' dtype), d <= 64, any chunk size.
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
// reverse. For b <= 64 every matrix of a chunk sits in shared memory; longer
// chunks are walked in blocks (linear_bwd_wide_kernel). Every product is a
// plain fp32 loop spread over the CTA's threads: the general form, for the
// 1e-4 bar of fp32 operands and the shapes linear_bwd_mma.cu does not take.
#include <algorithm>

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

// Chunks longer than 64 tokens (the large-chunk regime): the same recurrence,
// with a chunk walked in blocks of kSub tokens. E and dE of the chunk live in
// the workspace; S = tril(Q_c K_c^T) and P = -eta tril(dZ_c E^T) are formed one
// kSub x kSub block at a time, only on and below the diagonal, and applied at
// once: the sums over later (dE, dK) or earlier (dQ) tokens of the chunk run
// over blocks, the block's own entries masked by absolute token index.
constexpr int kSub = 32;

template <typename Tin>
__global__ void __launch_bounds__(kBwdThreads) linear_bwd_wide_kernel(LinearBwdParams p) {
  extern __shared__ __align__(16) float bsm[];
  const int d = p.d, b = p.b, T = p.T;
  const int unit = blockIdx.x;
  const int h = unit % p.H;
  const int tid = threadIdx.x;
  const float eta = p.eta[h];
  const int nch = (T + b - 1) / b;
  const int cap = min(b, T);     // tokens of the longest chunk
  float* W = bsm;                // [d][d]   chunk-start state
  float* G = W + d * d;          // [d][d]   gradient of the next chunk's start state
  float* R1 = G + d * d;         // [kSub][d] operands of the row block (tokens t)
  float* R2 = R1 + kSub * d;
  float* C1 = R2 + kSub * d;     // [kSub][d] operands of the column block (tokens t2)
  float* C2 = C1 + kSub * d;
  float* Acc = C2 + kSub * d;    // [kSub][d] the row block's result
  float* Sb = Acc + kSub * d;    // [kSub][kSub] one block of S or P
  float* red = Sb + kSub * kSub; // [kBwdThreads]
  const size_t base = static_cast<size_t>(unit) * T * d;
  float* states = p.states + static_cast<size_t>(unit) * nch * d * d;
  float* Ec = p.chunk_buf + static_cast<size_t>(unit) * 2 * cap * d;  // [cap][d]
  float* dEc = Ec + static_cast<size_t>(cap) * d;                      // [cap][d]

  auto load = [&](float* dst, const void* src, size_t off, int m) {
    for (int x = tid; x < m * d; x += kBwdThreads) dst[x] = ldv<Tin>(src, off + x);
  };
  auto load_ws = [&](float* dst, const float* src, int m) {
    for (int x = tid; x < m * d; x += kBwdThreads) dst[x] = src[x];
  };
  // Ec = K_c W - V_c for the n tokens of the chunk at `off`.
  auto chunk_errors = [&](size_t off, int n) {
    for (int r0 = 0; r0 < n; r0 += kSub) {
      const int m = min(kSub, n - r0);
      load(R1, p.K, off + static_cast<size_t>(r0) * d, m);
      load(R2, p.V, off + static_cast<size_t>(r0) * d, m);
      __syncthreads();
      for (int x = tid; x < m * d; x += kBwdThreads) {
        const int t = x / d, j = x % d;
        float acc = -R2[x];
        for (int k = 0; k < d; ++k) acc = fmaf(R1[t * d + k], W[k * d + j], acc);
        Ec[r0 * d + x] = acc;
      }
      __syncthreads();
    }
  };

  // ---------------------------------------------------------------- forward: chunk-start states
  for (int i = tid; i < d * d; i += kBwdThreads) W[i] = p.W0[static_cast<size_t>(h) * d * d + i];
  __syncthreads();
  for (int c = 0; c < nch; ++c) {
    const int c0 = c * b, n = min(b, T - c0);
    const size_t off = base + static_cast<size_t>(c0) * d;
    for (int i = tid; i < d * d; i += kBwdThreads) states[static_cast<size_t>(c) * d * d + i] = W[i];
    chunk_errors(off, n);
    for (int r0 = 0; r0 < n; r0 += kSub) {  // W -= eta K_c^T E, block by block
      const int m = min(kSub, n - r0);
      load(R1, p.K, off + static_cast<size_t>(r0) * d, m);
      load_ws(R2, Ec + r0 * d, m);
      __syncthreads();
      for (int x = tid; x < d * d; x += kBwdThreads) {
        const int i = x / d, j = x % d;
        float acc = 0.f;
        for (int t = 0; t < m; ++t) acc = fmaf(R1[t * d + i], R2[t * d + j], acc);
        W[x] -= eta * acc;
      }
      __syncthreads();
    }
  }

  // ---------------------------------------------------------------- backward, last chunk first
  for (int i = tid; i < d * d; i += kBwdThreads) G[i] = p.dW_out[static_cast<size_t>(unit) * d * d + i];
  float deta = 0.f;
  __syncthreads();
  for (int c = nch - 1; c >= 0; --c) {
    const int c0 = c * b, n = min(b, T - c0);
    const size_t off = base + static_cast<size_t>(c0) * d;
    for (int i = tid; i < d * d; i += kBwdThreads) W[i] = states[static_cast<size_t>(c) * d * d + i];
    __syncthreads();
    chunk_errors(off, n);

    // dE_t = -eta (k_t G + sum_{t2 >= t} (q_t2 . k_t) dz_t2); d eta -= E . (K G)
    for (int r0 = 0; r0 < n; r0 += kSub) {
      const int m = min(kSub, n - r0);
      load(R1, p.K, off + static_cast<size_t>(r0) * d, m);
      __syncthreads();
      for (int x = tid; x < m * d; x += kBwdThreads) {
        const int t = x / d, j = x % d;
        float kg = 0.f;
        for (int k = 0; k < d; ++k) kg = fmaf(R1[t * d + k], G[k * d + j], kg);
        deta -= Ec[r0 * d + x] * kg;
        Acc[x] = kg;
      }
      for (int q0 = r0; q0 < n; q0 += kSub) {
        const int mq = min(kSub, n - q0);
        load(C1, p.Q, off + static_cast<size_t>(q0) * d, mq);
        load(C2, p.dZ, off + static_cast<size_t>(q0) * d, mq);
        __syncthreads();
        for (int x = tid; x < mq * m; x += kBwdThreads) {  // Sb[t2][t] = q_t2 . k_t for t2 >= t
          const int t2 = x / m, t = x % m;
          float s = 0.f;
          if (q0 + t2 >= r0 + t)
            for (int k = 0; k < d; ++k) s = fmaf(C1[t2 * d + k], R1[t * d + k], s);
          Sb[t2 * kSub + t] = s;
        }
        __syncthreads();
        for (int x = tid; x < m * d; x += kBwdThreads) {
          const int t = x / d, j = x % d;
          float acc = Acc[x];
          for (int t2 = 0; t2 < mq; ++t2) acc = fmaf(Sb[t2 * kSub + t], C2[t2 * d + j], acc);
          Acc[x] = acc;
        }
        __syncthreads();
      }
      for (int x = tid; x < m * d; x += kBwdThreads) dEc[r0 * d + x] = -eta * Acc[x];
      __syncthreads();
    }

    // dQ_t = dz_t W^T + sum_{t2 <= t} P[t][t2] k_t2, P[t][t2] = -eta dz_t . e_t2;
    // d eta -= sum_{t2 <= t} (q_t . k_t2)(dz_t . e_t2)
    for (int r0 = 0; r0 < n; r0 += kSub) {
      const int m = min(kSub, n - r0);
      load(R1, p.dZ, off + static_cast<size_t>(r0) * d, m);
      load(R2, p.Q, off + static_cast<size_t>(r0) * d, m);
      __syncthreads();
      for (int x = tid; x < m * d; x += kBwdThreads) {
        const int t = x / d, i = x % d;
        float acc = 0.f;
        for (int j = 0; j < d; ++j) acc = fmaf(R1[t * d + j], W[i * d + j], acc);
        Acc[x] = acc;
      }
      for (int k0 = 0; k0 <= r0; k0 += kSub) {
        const int mk = min(kSub, n - k0);
        load_ws(C1, Ec + k0 * d, mk);
        load(C2, p.K, off + static_cast<size_t>(k0) * d, mk);
        __syncthreads();
        for (int x = tid; x < m * mk; x += kBwdThreads) {
          const int t = x / mk, t2 = x % mk;
          float pv = 0.f;
          if (k0 + t2 <= r0 + t) {
            float s = 0.f;
            for (int j = 0; j < d; ++j) {
              pv = fmaf(R1[t * d + j], C1[t2 * d + j], pv);
              s = fmaf(R2[t * d + j], C2[t2 * d + j], s);
            }
            deta -= s * pv;
          }
          Sb[t * kSub + t2] = -eta * pv;
        }
        __syncthreads();
        for (int x = tid; x < m * d; x += kBwdThreads) {
          const int t = x / d, i = x % d;
          float acc = Acc[x];
          for (int t2 = 0; t2 < mk; ++t2) acc = fmaf(Sb[t * kSub + t2], C2[t2 * d + i], acc);
          Acc[x] = acc;
        }
        __syncthreads();
      }
      for (int x = tid; x < m * d; x += kBwdThreads) stv<Tin>(p.dQ, off + static_cast<size_t>(r0) * d + x, Acc[x]);
      __syncthreads();
    }

    // dK_t = dE_t W^T - eta e_t G^T + sum_{t2 >= t} P[t2][t] q_t2;  dV = -dE
    for (int r0 = 0; r0 < n; r0 += kSub) {
      const int m = min(kSub, n - r0);
      load_ws(R1, dEc + r0 * d, m);
      load_ws(R2, Ec + r0 * d, m);
      __syncthreads();
      for (int x = tid; x < m * d; x += kBwdThreads) {
        const int t = x / d, i = x % d;
        float ak = 0.f, eg = 0.f;
        for (int j = 0; j < d; ++j) {
          ak = fmaf(R1[t * d + j], W[i * d + j], ak);
          eg = fmaf(R2[t * d + j], G[i * d + j], eg);
        }
        Acc[x] = ak - eta * eg;
        stv<Tin>(p.dV, off + static_cast<size_t>(r0) * d + x, -R1[x]);
      }
      for (int q0 = r0; q0 < n; q0 += kSub) {
        const int mq = min(kSub, n - q0);
        load(C1, p.dZ, off + static_cast<size_t>(q0) * d, mq);
        load(C2, p.Q, off + static_cast<size_t>(q0) * d, mq);
        __syncthreads();
        for (int x = tid; x < mq * m; x += kBwdThreads) {  // Sb[t2][t] = P[t2][t] for t2 >= t
          const int t2 = x / m, t = x % m;
          float pv = 0.f;
          if (q0 + t2 >= r0 + t)
            for (int j = 0; j < d; ++j) pv = fmaf(C1[t2 * d + j], R2[t * d + j], pv);
          Sb[t2 * kSub + t] = -eta * pv;
        }
        __syncthreads();
        for (int x = tid; x < m * d; x += kBwdThreads) {
          const int t = x / d, i = x % d;
          float acc = Acc[x];
          for (int t2 = 0; t2 < mq; ++t2) acc = fmaf(Sb[t2 * kSub + t], C2[t2 * d + i], acc);
          Acc[x] = acc;
        }
        __syncthreads();
      }
      for (int x = tid; x < m * d; x += kBwdThreads) stv<Tin>(p.dK, off + static_cast<size_t>(r0) * d + x, Acc[x]);
      __syncthreads();
    }

    // G += Q_c^T dZ_c + K_c^T dE (G was last read above)
    for (int r0 = 0; r0 < n; r0 += kSub) {
      const int m = min(kSub, n - r0);
      load(R1, p.Q, off + static_cast<size_t>(r0) * d, m);
      load(R2, p.dZ, off + static_cast<size_t>(r0) * d, m);
      load(C1, p.K, off + static_cast<size_t>(r0) * d, m);
      load_ws(C2, dEc + r0 * d, m);
      __syncthreads();
      for (int x = tid; x < d * d; x += kBwdThreads) {
        const int i = x / d, j = x % d;
        float acc = 0.f;
        for (int t = 0; t < m; ++t) acc = fmaf(R1[t * d + i], R2[t * d + j], fmaf(C1[t * d + i], C2[t * d + j], acc));
        G[x] += acc;
      }
      __syncthreads();
    }
  }

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

// dW0[h] and d eta[h]: sums over the batch rows (and segments) of the per-unit partials.
// Blocks: (head, slice of 256 of the d*d + 1 entries); one thread per entry.
__global__ void __launch_bounds__(kBwdThreads) linear_bwd_reduce_kernel(LinearBwdParams p) {
  const int d = p.d;
  const int n_ent = d * d + 1;
  const int slices = (n_ent + kBwdThreads - 1) / kBwdThreads;
  const int h = blockIdx.x / slices;
  const int i = (blockIdx.x % slices) * kBwdThreads + threadIdx.x;
  if (i >= n_ent) return;
  const int S = p.bseg_count > 1 ? p.bseg_count : 1;
  float acc = 0.f;
  for (int n = 0; n < p.B; ++n)
    for (int s = 0; s < S; ++s) acc += p.partial[(static_cast<size_t>(n * p.H + h) * S + s) * n_ent + i];
  if (i < d * d)
    p.dW0[static_cast<size_t>(h) * d * d + i] = acc;
  else
    p.deta[h] = acc;
}

}  // namespace

size_t linear_bwd_smem_bytes(int d, int b) {
  return (static_cast<size_t>(2) * d * d + static_cast<size_t>(7) * b * d + static_cast<size_t>(2) * b * b +
          kBwdThreads) *
         sizeof(float);
}

static size_t wide_smem_bytes(int d) {
  return (static_cast<size_t>(2) * d * d + static_cast<size_t>(5) * kSub * d + kSub * kSub + kBwdThreads) *
         sizeof(float);
}

static bool short_chunks(int d, int b) { return b <= 64 && linear_bwd_smem_bytes(d, b) <= 227 * 1024; }

bool linear_bwd_supported(int d, int b) { return d >= 1 && d <= 64 && b >= 1; }

size_t linear_bwd_scratch_bytes(int units, int T, int d, int b) {
  const size_t nch = (static_cast<size_t>(T) + b - 1) / b;
  size_t bytes = static_cast<size_t>(units) * nch * d * d * sizeof(float) +
                 static_cast<size_t>(units) * (static_cast<size_t>(d) * d + 1) * sizeof(float);
  if (!short_chunks(d, b))  // E and dE of one chunk per unit
    bytes += static_cast<size_t>(units) * 2 * std::min(b, T) * d * sizeof(float);
  return bytes;
}

float* linear_bwd_chunk_buf(float* partial, int units, int d) {
  return partial + static_cast<size_t>(units) * (static_cast<size_t>(d) * d + 1);
}

cudaError_t launch_linear_bwd(const LinearBwdParams& p, cudaStream_t stream) {
  const bool wide = !short_chunks(p.d, p.b);
  const size_t smem = wide ? wide_smem_bytes(p.d) : linear_bwd_smem_bytes(p.d, p.b);
  auto kern = wide ? (p.bf16 ? linear_bwd_wide_kernel<__nv_bfloat16> : linear_bwd_wide_kernel<float>)
                   : (p.bf16 ? linear_bwd_kernel<__nv_bfloat16> : linear_bwd_kernel<float>);
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  kern<<<p.units, kBwdThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_linear_bwd_reduce(const LinearBwdParams& p, cudaStream_t stream) {
  const int slices = (p.d * p.d + 1 + kBwdThreads - 1) / kBwdThreads;
  linear_bwd_reduce_kernel<<<p.H * slices, kBwdThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace ttt
