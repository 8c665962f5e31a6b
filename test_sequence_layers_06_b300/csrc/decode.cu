// TTT-Linear decode: N tokens per (batch row, head) in one launch, O(d^2) work
// and memory per token ("Test-Time Training (TTT) guide", section 3: constant
// time and memory per decoded token).
//
// The pair (W_anchor, W_run) is the chunk-start and the running state, so a
// token inside a chunk still takes its gradient at the chunk-start weights:
//   e = k W_anchor - v;  W_run <- W_run - eta k^T e;  z = q W_run
// and z is formed from the old W_run as q W_run - eta (q . k) e, so the read
// does not wait for the write. When a token completes a chunk, W_anchor takes
// the new W_run.
//
// Every one of these is a function of one output column j of the state, so a
// head's d columns are split over CTAs of 16 columns (4 CTAs per head at
// d = 64). A CTA holds its columns of W_anchor and W_run in registers for all
// N tokens: thread (i, c) keeps row i, columns 4c .. 4c + 3 of the slice of each
// state. Per token the column sums over i are a shuffle reduction within each
// warp plus a sum of the warps' partials in shared memory. The tokens' q, k and
// v are staged in shared memory 32 at a time; a launch of more than 32 tokens
// loads the next 32 into registers while the current ones are processed.
#include "kernels.h"
#include "ttt_device.cuh"

namespace ttt {
namespace {

constexpr int kCols = 16;                   // state columns per CTA
constexpr int kMaxD = 64;
constexpr int kThreads = kMaxD * kCols / 4;  // one float4 of each state per thread at d = 64
constexpr int kWarpsD = kThreads / 32;
constexpr int kTokBuf = 32;                 // tokens whose q, k, v are staged at once

template <typename T>
__device__ __forceinline__ float ld(const T* p);
template <>
__device__ __forceinline__ float ld<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ld<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }

template <typename T, bool kPrefetch>
__global__ void __launch_bounds__(kThreads) linear_decode_kernel(DecodeParams p) {
  __shared__ float qs[kTokBuf][kMaxD], ks[kTokBuf][kMaxD], vs[kTokBuf][kCols];
  __shared__ float part[2][kWarpsD][kCols];  // per-warp column sums of k W_anchor and q W_run
  __shared__ float es[kCols];
  __shared__ float qk[kTokBuf];
  const int groups = (p.d + kCols - 1) / kCols;
  const int unit = blockIdx.x / groups;
  const int j0 = (blockIdx.x % groups) * kCols;
  const int h = unit % p.H;
  const int d = p.d;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int i = tid >> 2;        // state row
  const int c = (tid & 3) * 4;   // first of this thread's 4 columns within the slice
  const bool row_ok = i < d;
  const float eta = p.eta[h];
  float* Wa = p.W_anchor + static_cast<size_t>(unit) * d * d;
  float* Wr = p.W_run + static_cast<size_t>(unit) * d * d;

  // This thread's 4 columns of row i (fewer at the right edge when d % 16 != 0).
  float wa[4] = {0.f, 0.f, 0.f, 0.f}, wr[4] = {0.f, 0.f, 0.f, 0.f};
  auto col_ok = [&](int q) { return row_ok && j0 + c + q < d; };
#pragma unroll
  for (int q = 0; q < 4; ++q)
    if (col_ok(q)) {
      wa[q] = Wa[i * d + j0 + c + q];
      wr[q] = Wr[i * d + j0 + c + q];
    }

  // With more than one batch of tokens (kPrefetch), a batch's q, k and v go through registers: the
  // next batch's loads are issued before the current batch's tokens are processed. A launch of one
  // batch stages directly (its code stays small: a one-token step is bound by its launch).
  constexpr int kPerQK = kPrefetch ? kTokBuf * kMaxD / kThreads : 1;
  constexpr int kPerV = kPrefetch ? kTokBuf * kCols / kThreads : 1;
  float rq[kPerQK], rk[kPerQK], rv[kPerV];
  auto fetch = [&](int n0) {
    const int nb = min(kTokBuf, p.N - n0);
#pragma unroll
    for (int y = 0; y < kPerQK; ++y) {
      const int x = tid + y * kThreads, t = x / kMaxD, f = x % kMaxD;
      rq[y] = rk[y] = 0.f;
      if (t < nb && f < d) {
        const size_t g = (static_cast<size_t>(unit) * p.N + n0 + t) * d + f;
        rq[y] = ld<T>(static_cast<const T*>(p.q) + g);
        rk[y] = ld<T>(static_cast<const T*>(p.k) + g);
      }
    }
#pragma unroll
    for (int y = 0; y < kPerV; ++y) {
      const int x = tid + y * kThreads, t = x / kCols, f = x % kCols;
      rv[y] = 0.f;
      if (t < nb && j0 + f < d)
        rv[y] = ld<T>(static_cast<const T*>(p.v) + (static_cast<size_t>(unit) * p.N + n0 + t) * d + j0 + f);
    }
  };
  if constexpr (kPrefetch) {
    if (p.N > 0) fetch(0);
  }
  for (int n0 = 0; n0 < p.N; n0 += kTokBuf) {
    const int nb = min(kTokBuf, p.N - n0);
    if constexpr (kPrefetch) {
      // Stage this batch (zeros past d and past the last token), then fetch the next one.
#pragma unroll
      for (int y = 0; y < kPerQK; ++y) {
        const int x = tid + y * kThreads;
        qs[x / kMaxD][x % kMaxD] = rq[y];
        ks[x / kMaxD][x % kMaxD] = rk[y];
      }
#pragma unroll
      for (int y = 0; y < kPerV; ++y) {
        const int x = tid + y * kThreads;
        vs[x / kCols][x % kCols] = rv[y];
      }
      __syncthreads();
      if (n0 + kTokBuf < p.N) fetch(n0 + kTokBuf);
    } else {
      // Stage the q, k (all d) and v (this slice) of the next nb tokens.
      for (int x = tid; x < nb * d; x += kThreads) {
        const int t = x / d, f = x % d;
        const size_t g = (static_cast<size_t>(unit) * p.N + n0 + t) * d + f;
        qs[t][f] = ld<T>(static_cast<const T*>(p.q) + g);
        ks[t][f] = ld<T>(static_cast<const T*>(p.k) + g);
        if (f >= j0 && f < j0 + kCols) vs[t][f - j0] = ld<T>(static_cast<const T*>(p.v) + g);
      }
      __syncthreads();
    }
    for (int t = warp; t < nb; t += kWarpsD) {  // q . k per token, a warp each
      float s = 0.f;
      for (int f = lane; f < d; f += 32) s = fmaf(qs[t][f], ks[t][f], s);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (lane == 0) qk[t] = s;
    }
    for (int t = 0; t < nb; ++t) {
      const float kv = row_ok ? ks[t][i] : 0.f, qv = row_ok ? qs[t][i] : 0.f;
      float se[4], sz[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        se[q] = kv * wa[q];
        sz[q] = qv * wr[q];
      }
      // sum over the warp's 8 rows (lanes with equal lane % 4 hold the same columns)
#pragma unroll
      for (int o = 4; o < 32; o <<= 1)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          se[q] += __shfl_xor_sync(0xffffffffu, se[q], o);
          sz[q] += __shfl_xor_sync(0xffffffffu, sz[q], o);
        }
      if (lane < 4)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          part[0][warp][4 * lane + q] = se[q];
          part[1][warp][4 * lane + q] = sz[q];
        }
      __syncthreads();
      if (tid < kCols) {
        float a = 0.f, z = 0.f;
#pragma unroll
        for (int w = 0; w < kWarpsD; ++w) {
          a += part[0][w][tid];
          z += part[1][w][tid];
        }
        const float e = a - vs[t][tid];
        es[tid] = e;
        if (j0 + tid < d) {
          const size_t o = (static_cast<size_t>(unit) * p.N + n0 + t) * d + j0 + tid;
          const float zz = z - eta * qk[t] * e;
          if (p.bf16)
            static_cast<__nv_bfloat16*>(p.z)[o] = __float2bfloat16_rn(zz);
          else
            static_cast<float*>(p.z)[o] = zz;
        }
      }
      __syncthreads();
      const bool completes = ((p.pos + n0 + t + 1) % p.b) == 0;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        wr[q] -= eta * kv * es[c + q];
        if (completes) wa[q] = wr[q];
      }
    }
    __syncthreads();  // the staged tokens are read; the next batch may overwrite them
  }
#pragma unroll
  for (int q = 0; q < 4; ++q)
    if (col_ok(q)) {
      Wa[i * d + j0 + c + q] = wa[q];
      Wr[i * d + j0 + c + q] = wr[q];
    }
}

}  // namespace

cudaError_t launch_linear_decode(const DecodeParams& p, cudaStream_t stream) {
  if (p.units == 0 || p.N == 0) return cudaSuccess;
  const int grid = p.units * ((p.d + kCols - 1) / kCols);
  const bool many = p.N > kTokBuf;
  if (p.bf16) {
    if (many)
      linear_decode_kernel<__nv_bfloat16, true><<<grid, kThreads, 0, stream>>>(p);
    else
      linear_decode_kernel<__nv_bfloat16, false><<<grid, kThreads, 0, stream>>>(p);
  } else {
    if (many)
      linear_decode_kernel<float, true><<<grid, kThreads, 0, stream>>>(p);
    else
      linear_decode_kernel<float, false><<<grid, kThreads, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace ttt
