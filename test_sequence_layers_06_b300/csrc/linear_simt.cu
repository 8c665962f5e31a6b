// TTT-Linear forward in plain fp32 arithmetic for any d <= 64, any chunk size b
// and fp32 or bf16 inputs: the path for fp32 operands (whose tolerance rules
// out bf16 tensor-core products) and for shapes the tensor-core kernel does
// not take. One CTA per (batch row, head); the state lives in shared memory.
//
// Method ("5 · TestingTime 训练与长上下文", sections 1.1 and 2.3): per chunk,
// with Wa its start state, E = K Wa - V, Z = Q Wa - eta tril(Q K^T) E,
// W = Wa - eta K^T E. The chunk is walked in pieces of at most 16 tokens that
// never cross a chunk boundary; a piece reads out with the running W (which
// holds the gradients of the chunk's earlier pieces) plus its own tril term,
// which is the same product split by rows.
#include "kernels.h"
#include "ttt_device.cuh"

namespace ttt {
namespace {

constexpr int kPiece = 16;
constexpr int kThreads = 256;

template <typename T>
__device__ __forceinline__ float load_in(const T* p);
template <>
__device__ __forceinline__ float load_in<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float load_in<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }

template <typename T>
__device__ __forceinline__ void store_out(T* p, float v);
template <>
__device__ __forceinline__ void store_out<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void store_out<__nv_bfloat16>(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

template <typename T>
__global__ void __launch_bounds__(kThreads) linear_simt_kernel(LinearParams p) {
  extern __shared__ float sm[];
  const int d = p.d;
  float* Wr = sm;               // running state [d][d]
  float* Wa = Wr + d * d;       // chunk-start state [d][d]
  float* Qs = Wa + d * d;       // [16][d]
  float* Ks = Qs + kPiece * d;
  float* Vs = Ks + kPiece * d;
  float* Es = Vs + kPiece * d;
  float* Ss = Es + kPiece * d;  // [16][16]

  const int unit = blockIdx.x;
  const int h = unit % p.H;
  const int tid = threadIdx.x;
  const float eta = p.eta[h];
  const size_t base = static_cast<size_t>(unit) * p.T * d;
  const T* Q = static_cast<const T*>(p.Q) + base;
  const T* K = static_cast<const T*>(p.K) + base;
  const T* V = static_cast<const T*>(p.V) + base;
  T* Z = static_cast<T*>(p.Z) + base;

  const float* W0 = p.W0 + static_cast<size_t>(h) * d * d;
  for (int x = tid; x < d * d; x += kThreads) Wr[x] = Wa[x] = W0[x];
  __syncthreads();

  for (int t0 = 0; t0 < p.T;) {
    const int chunk_end = min((t0 / p.b + 1) * p.b, p.T);
    const int t1 = min(t0 + kPiece, chunk_end);
    const int n = t1 - t0;
    for (int x = tid; x < n * d; x += kThreads) {
      const size_t g = static_cast<size_t>(t0) * d + x;
      Qs[x] = load_in<T>(Q + g);
      Ks[x] = load_in<T>(K + g);
      Vs[x] = load_in<T>(V + g);
    }
    __syncthreads();
    // E = K Wa - V; S = tril(Q K^T)
    for (int x = tid; x < n * d; x += kThreads) {
      const int t = x / d, j = x % d;
      float s = 0.f;
      for (int i = 0; i < d; ++i) s = fmaf(Ks[t * d + i], Wa[i * d + j], s);
      Es[x] = s - Vs[x];
    }
    for (int x = tid; x < n * n; x += kThreads) {
      const int t = x / n, t2 = x % n;
      float s = 0.f;
      if (t2 <= t)
        for (int i = 0; i < d; ++i) s = fmaf(Qs[t * d + i], Ks[t2 * d + i], s);
      Ss[t * kPiece + t2] = s;
    }
    __syncthreads();
    // Z = Q W_run - eta S E
    for (int x = tid; x < n * d; x += kThreads) {
      const int t = x / d, j = x % d;
      float qw = 0.f, se = 0.f;
      for (int i = 0; i < d; ++i) qw = fmaf(Qs[t * d + i], Wr[i * d + j], qw);
      for (int t2 = 0; t2 <= t; ++t2) se = fmaf(Ss[t * kPiece + t2], Es[t2 * d + j], se);
      store_out<T>(Z + static_cast<size_t>(t0) * d + x, qw - eta * se);
    }
    __syncthreads();
    // W_run -= eta K^T E
    for (int x = tid; x < d * d; x += kThreads) {
      const int i = x / d, j = x % d;
      float s = 0.f;
      for (int t = 0; t < n; ++t) s = fmaf(Ks[t * d + i], Es[t * d + j], s);
      Wr[x] -= eta * s;
    }
    __syncthreads();
    if (t1 == chunk_end) {
      for (int x = tid; x < d * d; x += kThreads) Wa[x] = Wr[x];
      __syncthreads();
    }
    t0 = t1;
  }
  float* Wo = p.W_out + static_cast<size_t>(unit) * d * d;
  for (int x = tid; x < d * d; x += kThreads) Wo[x] = Wr[x];
}

}  // namespace

cudaError_t launch_linear_simt(const LinearParams& p, cudaStream_t stream) {
  if (p.units == 0) return cudaSuccess;
  const size_t smem = sizeof(float) * (2 * p.d * p.d + 4 * kPiece * p.d + kPiece * kPiece);
  cudaError_t err;
  if (p.bf16) {
    err = cudaFuncSetAttribute(linear_simt_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    linear_simt_kernel<__nv_bfloat16><<<p.units, kThreads, smem, stream>>>(p);
  } else {
    err = cudaFuncSetAttribute(linear_simt_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    linear_simt_kernel<float><<<p.units, kThreads, smem, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace ttt
