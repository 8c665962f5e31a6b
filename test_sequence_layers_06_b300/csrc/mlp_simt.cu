// TTT-MLP forward in plain fp32 arithmetic (any dtype, d <= 64, hidden m,
// any b): the path for fp32 operands and for shapes the tensor-core kernel
// (mlp_mma.cu) does not take. f(x) = gelu(x W1) W2 with tanh-GELU ("Test-Time Training (TTT)
// guide", section 3: two layers, hidden 4x, GELU; it stores the hidden
// activations, so it moves more memory than TTT-Linear).
//
// Per chunk with start weights W1a, W2a, in dual form:
//   U = K W1a, A = gelu(U), G = A W2a - V, D = (G W2a^T) .* gelu'(U)
//   Hq = Q W1a - eta tril(Q K^T) D,  Aq = gelu(Hq)
//   Z = Aq W2a - eta tril(Aq A^T) G
//   W1 = W1a - eta K^T D,  W2 = W2a - eta A^T G
// walked in pieces of at most 16 tokens (running weights for the read-out, as
// in the TTT-Linear kernels). The running state lives in W1_out / W2_out and
// the chunk-start snapshot in the workspace; both stay in L2.
#include "kernels.h"
#include "ttt_device.cuh"

namespace ttt {
namespace {

constexpr int kPiece = 16;
constexpr int kThreads = 256;

template <typename T>
__device__ __forceinline__ float ldv(const T* p);
template <>
__device__ __forceinline__ float ldv<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ldv<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }

__device__ __forceinline__ void gelu_and_prime(float u, float* g, float* gp) {
  const float c = 0.7978845608028654f;  // sqrt(2/pi)
  const float a = 0.044715f;
  const float th = tanhf(c * (u + a * u * u * u));
  *g = 0.5f * u * (1.f + th);
  if (gp) *gp = 0.5f * (1.f + th) + 0.5f * u * (1.f - th * th) * c * (1.f + 3.f * a * u * u);
}

template <typename T>
__global__ void __launch_bounds__(kThreads) mlp_simt_kernel(MlpParams p) {
  extern __shared__ float sm[];
  const int d = p.d, m = p.m;
  float* Qs = sm;                 // [16][d]
  float* Ks = Qs + kPiece * d;
  float* Vs = Ks + kPiece * d;
  float* Gs = Vs + kPiece * d;    // [16][d]
  float* As = Gs + kPiece * d;    // [16][m]  gelu(U)
  float* Ps = As + kPiece * m;    // [16][m]  gelu'(U), then reused for Aq
  float* Ds = Ps + kPiece * m;    // [16][m]
  float* Sq = Ds + kPiece * m;    // [16][16] tril(Q K^T)
  float* Sa = Sq + kPiece * kPiece;  // [16][16] tril(Aq A^T)

  const int unit = blockIdx.x;
  const int h = unit % p.H;
  const int tid = threadIdx.x;
  const float eta = p.eta[h];
  const size_t base = static_cast<size_t>(unit) * p.T * d;
  const T* Q = static_cast<const T*>(p.Q) + base;
  const T* K = static_cast<const T*>(p.K) + base;
  const T* V = static_cast<const T*>(p.V) + base;
  T* Z = static_cast<T*>(p.Z) + base;
  float* W1 = p.W1_out + static_cast<size_t>(unit) * d * m;
  float* W2 = p.W2_out + static_cast<size_t>(unit) * m * d;
  float* W1a = p.snap + static_cast<size_t>(unit) * 2 * d * m;
  float* W2a = W1a + static_cast<size_t>(d) * m;
  const float* W10 = p.W1_0 + static_cast<size_t>(h) * d * m;
  const float* W20 = p.W2_0 + static_cast<size_t>(h) * m * d;
  for (int x = tid; x < d * m; x += kThreads) {
    W1[x] = W1a[x] = W10[x];
    W2[x] = W2a[x] = W20[x];
  }
  __syncthreads();

  for (int t0 = 0; t0 < p.T;) {
    const int chunk_end = min((t0 / p.b + 1) * p.b, p.T);
    const int t1 = min(t0 + kPiece, chunk_end);
    const int n = t1 - t0;
    for (int x = tid; x < n * d; x += kThreads) {
      const size_t g = static_cast<size_t>(t0) * d + x;
      Qs[x] = ldv<T>(Q + g);
      Ks[x] = ldv<T>(K + g);
      Vs[x] = ldv<T>(V + g);
    }
    __syncthreads();
    // U = K W1a; A = gelu(U); P = gelu'(U).   Sq = tril(Q K^T)
    for (int x = tid; x < n * m; x += kThreads) {
      const int t = x / m, c = x % m;
      float s = 0.f;
      for (int i = 0; i < d; ++i) s = fmaf(Ks[t * d + i], W1a[i * m + c], s);
      gelu_and_prime(s, &As[x], &Ps[x]);
    }
    for (int x = tid; x < n * n; x += kThreads) {
      const int t = x / n, t2 = x % n;
      float s = 0.f;
      if (t2 <= t)
        for (int i = 0; i < d; ++i) s = fmaf(Qs[t * d + i], Ks[t2 * d + i], s);
      Sq[t * kPiece + t2] = s;
    }
    __syncthreads();
    // G = A W2a - V
    for (int x = tid; x < n * d; x += kThreads) {
      const int t = x / d, j = x % d;
      float s = 0.f;
      for (int c = 0; c < m; ++c) s = fmaf(As[t * m + c], W2a[c * d + j], s);
      Gs[x] = s - Vs[x];
    }
    __syncthreads();
    // D = (G W2a^T) .* gelu'(U)
    for (int x = tid; x < n * m; x += kThreads) {
      const int t = x / m, c = x % m;
      float s = 0.f;
      for (int j = 0; j < d; ++j) s = fmaf(Gs[t * d + j], W2a[c * d + j], s);
      Ds[x] = s * Ps[x];
    }
    __syncthreads();
    // Aq = gelu(Q W1_run - eta Sq D)   (into Ps)
    for (int x = tid; x < n * m; x += kThreads) {
      const int t = x / m, c = x % m;
      float s = 0.f, r = 0.f;
      for (int i = 0; i < d; ++i) s = fmaf(Qs[t * d + i], W1[i * m + c], s);
      for (int t2 = 0; t2 <= t; ++t2) r = fmaf(Sq[t * kPiece + t2], Ds[t2 * m + c], r);
      gelu_and_prime(s - eta * r, &Ps[x], nullptr);
    }
    __syncthreads();
    // Sa = tril(Aq A^T)
    for (int x = tid; x < n * n; x += kThreads) {
      const int t = x / n, t2 = x % n;
      float s = 0.f;
      if (t2 <= t)
        for (int c = 0; c < m; ++c) s = fmaf(Ps[t * m + c], As[t2 * m + c], s);
      Sa[t * kPiece + t2] = s;
    }
    __syncthreads();
    // Z = Aq W2_run - eta Sa G
    for (int x = tid; x < n * d; x += kThreads) {
      const int t = x / d, j = x % d;
      float s = 0.f, r = 0.f;
      for (int c = 0; c < m; ++c) s = fmaf(Ps[t * m + c], W2[c * d + j], s);
      for (int t2 = 0; t2 <= t; ++t2) r = fmaf(Sa[t * kPiece + t2], Gs[t2 * d + j], r);
      const float zv = s - eta * r;
      if (p.bf16)
        reinterpret_cast<__nv_bfloat16*>(Z)[static_cast<size_t>(t0) * d + x] = __float2bfloat16_rn(zv);
      else
        reinterpret_cast<float*>(Z)[static_cast<size_t>(t0) * d + x] = zv;
    }
    __syncthreads();
    // W1 -= eta K^T D;  W2 -= eta A^T G
    for (int x = tid; x < d * m; x += kThreads) {
      const int i = x / m, c = x % m;
      float s = 0.f;
      for (int t = 0; t < n; ++t) s = fmaf(Ks[t * d + i], Ds[t * m + c], s);
      W1[x] -= eta * s;
    }
    for (int x = tid; x < m * d; x += kThreads) {
      const int c = x / d, j = x % d;
      float s = 0.f;
      for (int t = 0; t < n; ++t) s = fmaf(As[t * m + c], Gs[t * d + j], s);
      W2[x] -= eta * s;
    }
    __syncthreads();
    if (t1 == chunk_end) {
      for (int x = tid; x < d * m; x += kThreads) {
        W1a[x] = W1[x];
        W2a[x] = W2[x];
      }
      __syncthreads();
    }
    t0 = t1;
  }
}

}  // namespace

size_t mlp_simt_snapshot_bytes(int units, int d, int m) {
  return sizeof(float) * 2 * static_cast<size_t>(units) * d * m;
}

cudaError_t launch_mlp_simt(const MlpParams& p, cudaStream_t stream) {
  if (p.units == 0) return cudaSuccess;
  const size_t smem =
      sizeof(float) * (4 * kPiece * p.d + 3 * kPiece * p.m + 2 * kPiece * kPiece);
  cudaError_t err;
  if (p.bf16) {
    err = cudaFuncSetAttribute(mlp_simt_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    mlp_simt_kernel<__nv_bfloat16><<<p.units, kThreads, smem, stream>>>(p);
  } else {
    err = cudaFuncSetAttribute(mlp_simt_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    mlp_simt_kernel<float><<<p.units, kThreads, smem, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace ttt
