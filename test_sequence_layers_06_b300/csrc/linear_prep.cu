// Two inner-model variants of TTT-Linear on the tensor-core kernels, by changing
// their inputs (bf16 operands). Both are the plain chunk rule of the dual form
// ("5 · TestingTime 训练与长上下文", sections 1.1 and 3.1; "Test-Time Training
// (TTT) guide", section 3) on other Q, K, V and W0:
//
//   bias, f(k) = k W + beta (d <= 63): append a constant-1 feature to q and k,
//     pad every row to 64 features, and stack beta under W:
//       q' = [q | 1 | 0],  k' = [k | 1 | 0],  v' = [v | 0],  W0' = [[W0, 0]; [beta0, 0]; [0, 0]].
//     Then e' = k' W' - v' = [k W + beta - v | 0], the update of W' is the
//     updates of W (rows < d) and of beta (row d), the padded columns of W'
//     stay 0, and z' = q' W' = [q W + beta | 0].
//   learning rate per token, eta_t >= 0 (d <= 64): scale k and v by sqrt(eta_t)
//     and run with eta = 1, since sqrt(eta_t) k^T (sqrt(eta_t) k W - sqrt(eta_t) v)
//     = eta_t k^T (k W - v); q is unchanged (padded with zeros when d < 64).
//
// variant_prep_kernel writes the changed inputs (bf16, 64 features per row) and
// W0' (fp32); variant_post_kernel copies Z, W_out and beta_out back out of the
// padded results and merges the status words. Both are elementwise passes in which
// a thread handles 8 features of a padded row (16-byte loads of K and V where the
// rows are already 64 wide, element loads otherwise; 16-byte stores of the padded
// rows).
#include <algorithm>

#include "ttt_device.cuh"
#include "kernels.h"

namespace ttt {
namespace {

constexpr int kPrepThreads = 256;
constexpr int kP = 64;  // padded width

enum : int { kWhereNegativeRate = 20 };

__device__ __forceinline__ float ldbf(const void* p, size_t i) {
  return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
}

// Blocks [0, H): W0' and eta' of head h. Blocks from H on: token rows, one warp
// per row, grid-stride.
__global__ void __launch_bounds__(kPrepThreads) variant_prep_kernel(VariantPrepParams p) {
  const int d = p.d;
  if (static_cast<int>(blockIdx.x) < p.H) {
    const int h = blockIdx.x;
    for (int x = threadIdx.x; x < kP * kP; x += kPrepThreads) {
      const int i = x / kP, j = x % kP;
      float w = 0.f;
      if (i < d && j < d)
        w = p.W0[(static_cast<size_t>(h) * d + i) * d + j];
      else if (p.bias && i == d && j < d)
        w = p.beta0[static_cast<size_t>(h) * d + j];
      p.W0p[static_cast<size_t>(h) * kP * kP + x] = w;
    }
    if (threadIdx.x == 0) p.etap[h] = p.eta ? p.eta[h] : 1.f;
    return;
  }
  const long long rows = static_cast<long long>(p.units) * p.T;
  if (d == kP && !p.bias && p.Qp == nullptr) {
    // Rows of 64 features, 16-byte aligned: a thread scales 8 features of K and of V.
    const long long items = rows * (kP / 8);
    const long long stride = static_cast<long long>(gridDim.x - p.H) * kPrepThreads;
    for (long long x = static_cast<long long>(blockIdx.x - p.H) * kPrepThreads + threadIdx.x; x < items; x += stride) {
      const long long r = x / (kP / 8);
      float s = 1.f;
      if (p.tok_rate) {
        const float et = p.tok_rate[r];
        if (et < 0.f) {
          if ((x % (kP / 8)) == 0) report_error(p.status, TTT_ERR_DEVICE_CHECK, kWhereNegativeRate, static_cast<int>(r / p.T));
          s = 0.f;
        } else {
          s = sqrtf(et);
        }
      }
      const uint4 kv = reinterpret_cast<const uint4*>(p.K)[x];
      const uint4 vv = reinterpret_cast<const uint4*>(p.V)[x];
      const uint32_t ki[4] = {kv.x, kv.y, kv.z, kv.w}, vi[4] = {vv.x, vv.y, vv.z, vv.w};
      uint32_t ko[4], vo[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        ko[q] = pack_bf16(s * bf16_lo(ki[q]), s * bf16_hi(ki[q]));
        vo[q] = pack_bf16(s * bf16_lo(vi[q]), s * bf16_hi(vi[q]));
      }
      reinterpret_cast<uint4*>(p.Kp)[x] = make_uint4(ko[0], ko[1], ko[2], ko[3]);
      reinterpret_cast<uint4*>(p.Vp)[x] = make_uint4(vo[0], vo[1], vo[2], vo[3]);
    }
    return;
  }
  // Other widths (rows of d < 64 features, not 16-byte aligned): a thread forms 8 padded
  // features of a row from element loads and writes them as one 16-byte store.
  {
    const long long items = rows * (kP / 8);
    const long long stride = static_cast<long long>(gridDim.x - p.H) * kPrepThreads;
    for (long long x = static_cast<long long>(blockIdx.x - p.H) * kPrepThreads + threadIdx.x; x < items; x += stride) {
      const long long r = x / (kP / 8);
      const int f0 = static_cast<int>(x % (kP / 8)) * 8;
      float s = 1.f;
      if (p.tok_rate) {
        const float et = p.tok_rate[r];
        if (et < 0.f) {
          if (f0 == 0) report_error(p.status, TTT_ERR_DEVICE_CHECK, kWhereNegativeRate, static_cast<int>(r / p.T));
          s = 0.f;
        } else {
          s = sqrtf(et);
        }
      }
      const size_t in = static_cast<size_t>(r) * d;
      float q[8], k[8], v[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int f = f0 + e;
        const float one = (p.bias && f == d) ? 1.f : 0.f;
        q[e] = f < d ? ldbf(p.Q, in + f) : one;
        k[e] = f < d ? s * ldbf(p.K, in + f) : one;
        v[e] = f < d ? s * ldbf(p.V, in + f) : 0.f;
      }
      if (p.Qp)
        reinterpret_cast<uint4*>(p.Qp)[x] = make_uint4(pack_bf16(q[0], q[1]), pack_bf16(q[2], q[3]),
                                                       pack_bf16(q[4], q[5]), pack_bf16(q[6], q[7]));
      reinterpret_cast<uint4*>(p.Kp)[x] = make_uint4(pack_bf16(k[0], k[1]), pack_bf16(k[2], k[3]),
                                                     pack_bf16(k[4], k[5]), pack_bf16(k[6], k[7]));
      reinterpret_cast<uint4*>(p.Vp)[x] = make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]),
                                                     pack_bf16(v[4], v[5]), pack_bf16(v[6], v[7]));
    }
    return;
  }
}

// Blocks [0, units): W_out (and beta_out) of a unit from the padded state; block 0
// also merges the status word of the inner forward into the call's. Blocks from
// units on: Z rows, one warp per row, grid-stride.
__global__ void __launch_bounds__(kPrepThreads) variant_post_kernel(VariantPostParams p) {
  const int d = p.d;
  if (static_cast<int>(blockIdx.x) < p.units) {
    const int unit = blockIdx.x;
    if (unit == 0 && threadIdx.x == 0 && p.sub->code != 0) report_error(p.status, p.sub->code, p.sub->where, p.sub->unit);
    if (p.Wp == nullptr) return;
    const float* Wu = p.Wp + static_cast<size_t>(unit) * kP * kP;
    for (int x = threadIdx.x; x < d * d; x += kPrepThreads) {
      const int i = x / d, j = x % d;
      p.W_out[static_cast<size_t>(unit) * d * d + x] = Wu[i * kP + j];
    }
    if (p.beta_out)
      for (int j = threadIdx.x; j < d; j += kPrepThreads) p.beta_out[static_cast<size_t>(unit) * d + j] = Wu[d * kP + j];
    return;
  }
  if (p.Zp == nullptr) return;
  // A thread reads 8 padded features of a row as one 16-byte load and writes those below d.
  const long long rows = static_cast<long long>(p.units) * p.T;
  const long long items = rows * (kP / 8);
  const long long stride = static_cast<long long>(gridDim.x - p.units) * kPrepThreads;
  for (long long x = static_cast<long long>(blockIdx.x - p.units) * kPrepThreads + threadIdx.x; x < items; x += stride) {
    const long long r = x / (kP / 8);
    const int f0 = static_cast<int>(x % (kP / 8)) * 8;
    const uint4 zv = reinterpret_cast<const uint4*>(p.Zp)[x];
    const uint32_t zz[4] = {zv.x, zv.y, zv.z, zv.w};
    const size_t out = static_cast<size_t>(r) * d;
    __nv_bfloat16* Z = static_cast<__nv_bfloat16*>(p.Z);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int f = f0 + e;
      const uint16_t bits = static_cast<uint16_t>((e & 1) ? (zz[e >> 1] >> 16) : (zz[e >> 1] & 0xFFFFu));
      if (f < d) Z[out + f] = __ushort_as_bfloat16(bits);
    }
  }
}

int row_blocks(long long rows) {
  const long long want = (rows + kPrepThreads / 32 - 1) / (kPrepThreads / 32);
  return static_cast<int>(std::min<long long>(want, 148LL * 32));
}

}  // namespace

cudaError_t launch_variant_prep(const VariantPrepParams& p, cudaStream_t stream) {
  const long long rows = static_cast<long long>(p.units) * p.T;
  variant_prep_kernel<<<p.H + (rows > 0 ? row_blocks(rows) : 0), kPrepThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_variant_post(const VariantPostParams& p, cudaStream_t stream) {
  const long long rows = static_cast<long long>(p.units) * p.T;
  const int zblocks = (p.Zp != nullptr && rows > 0) ? row_blocks(rows) : 0;
  variant_post_kernel<<<p.units + zblocks, kPrepThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace ttt
