// TTT-Linear decode: one token per (batch row, head), O(d^2) work and memory
// per head ("Test-Time Training (TTT) guide", section 3: constant time and
// memory per decoded token).
//
// The pair (W_anchor, W_run) is the chunk-start and the running state, so a
// token inside a chunk still takes its gradient at the chunk-start weights:
//   e = k W_anchor - v;  W_run <- W_run - eta k^T e;  z = q W_run
// and z is formed from the old W_run as q W_run - eta (q . k) e, so the read
// does not wait for the write. When the token completes a chunk, W_anchor
// takes the new W_run.
#include "kernels.h"
#include "ttt_device.cuh"

namespace ttt {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxD = 64;
constexpr int kParts = kThreads / kMaxD;  // 4 partial sums per column

template <typename T>
__device__ __forceinline__ float ld(const T* p);
template <>
__device__ __forceinline__ float ld<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ld<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }

template <typename T>
__global__ void __launch_bounds__(kThreads) linear_decode_kernel(DecodeParams p) {
  __shared__ float qs[kMaxD], ks[kMaxD], vs[kMaxD], es[kMaxD];
  __shared__ float pe[kParts][kMaxD], pz[kParts][kMaxD];
  __shared__ float qk;
  const int unit = blockIdx.x;
  const int h = unit % p.H;
  const int d = p.d;
  const int tid = threadIdx.x;
  const float eta = p.eta[h];
  const T* q = static_cast<const T*>(p.q) + static_cast<size_t>(unit) * d;
  const T* k = static_cast<const T*>(p.k) + static_cast<size_t>(unit) * d;
  const T* v = static_cast<const T*>(p.v) + static_cast<size_t>(unit) * d;
  float* Wa = p.W_anchor + static_cast<size_t>(unit) * d * d;
  float* Wr = p.W_run + static_cast<size_t>(unit) * d * d;

  if (tid < d) {
    qs[tid] = ld<T>(q + tid);
    ks[tid] = ld<T>(k + tid);
    vs[tid] = ld<T>(v + tid);
  }
  __syncthreads();
  if (tid < 32) {
    float s = 0.f;
    for (int i = tid; i < d; i += 32) s = fmaf(qs[i], ks[i], s);
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (tid == 0) qk = s;
  }
  const int j = tid % kMaxD;
  const int part = tid / kMaxD;
  if (j < d) {
    float se = 0.f, sz = 0.f;
    for (int i = part; i < d; i += kParts) {
      se = fmaf(ks[i], Wa[i * d + j], se);
      sz = fmaf(qs[i], Wr[i * d + j], sz);
    }
    pe[part][j] = se;
    pz[part][j] = sz;
  }
  __syncthreads();
  if (tid < d) {
    float se = 0.f, sz = 0.f;
    for (int r = 0; r < kParts; ++r) {
      se += pe[r][tid];
      sz += pz[r][tid];
    }
    const float e = se - vs[tid];
    es[tid] = e;
    const float z = sz - eta * qk * e;
    if (p.bf16)
      static_cast<__nv_bfloat16*>(p.z)[static_cast<size_t>(unit) * d + tid] = __float2bfloat16_rn(z);
    else
      static_cast<float*>(p.z)[static_cast<size_t>(unit) * d + tid] = z;
  }
  __syncthreads();
  const bool completes = ((p.pos + 1) % p.b) == 0;
  for (int x = tid; x < d * d; x += kThreads) {
    const int i = x / d, jj = x % d;
    const float w = Wr[x] - eta * ks[i] * es[jj];
    Wr[x] = w;
    if (completes) Wa[x] = w;
  }
}

}  // namespace

cudaError_t launch_linear_decode(const DecodeParams& p, cudaStream_t stream) {
  if (p.units == 0) return cudaSuccess;
  if (p.bf16)
    linear_decode_kernel<__nv_bfloat16><<<p.units, kThreads, 0, stream>>>(p);
  else
    linear_decode_kernel<float><<<p.units, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace ttt
