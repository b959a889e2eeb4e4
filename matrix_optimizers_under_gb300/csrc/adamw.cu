// Fused AdamW over the packed non-matrix tail.
//
// MatrixFSDP: Communication-Free Matrix Optimizers Under ZeRO-3 Parameter
// Sharding -- Abstract: non-matrix tensors are packed into tail owners and stay
// on AdamW.  Decoupled weight decay (PyTorch order), bias corrections folded
// into scalars computed on the host in double precision.
//
// One pass over HBM: read p, g, m, v and write p, m, v (28 bytes per element),
// 128-bit streaming loads/stores, a grid-stride loop over a grid that is a
// multiple of the SM count, two float4 groups in flight per thread.
#include <algorithm>

#include "mfsdp_internal.h"

namespace mfsdp {
namespace {

__device__ __forceinline__ void adam1(float& p, float g, float& m, float& v, const AdamScalars& k) {
  p *= k.decay;
  m = fmaf(k.beta1, m, k.omb1 * g);
  v = fmaf(k.beta2, v, k.omb2 * g * g);
  const float denom = fmaf(sqrtf(v), k.inv_sqrt_bc2, k.eps);
  p = fmaf(-k.step_size, m / denom, p);
}

__device__ __forceinline__ void adam4(float4& p, const float4& g, float4& m, float4& v, const AdamScalars& k) {
  adam1(p.x, g.x, m.x, v.x, k);
  adam1(p.y, g.y, m.y, v.y, k);
  adam1(p.z, g.z, m.z, v.z, k);
  adam1(p.w, g.w, m.w, v.w, k);
}

__global__ void __launch_bounds__(256) adamw_kernel(float* __restrict__ p, const float* __restrict__ g,
                                                    float* __restrict__ m, float* __restrict__ v, int64_t n,
                                                    AdamScalars k) {
  const int64_t n4 = n >> 2;
  float4* p4 = reinterpret_cast<float4*>(p);
  const float4* g4 = reinterpret_cast<const float4*>(g);
  float4* m4 = reinterpret_cast<float4*>(m);
  float4* v4 = reinterpret_cast<float4*>(v);
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + stride < n4; i += 2 * stride) {
    float4 pa = __ldcs(p4 + i), pb = __ldcs(p4 + i + stride);
    const float4 ga = __ldcs(g4 + i), gb = __ldcs(g4 + i + stride);
    float4 ma = __ldcs(m4 + i), mb = __ldcs(m4 + i + stride);
    float4 va = __ldcs(v4 + i), vb = __ldcs(v4 + i + stride);
    adam4(pa, ga, ma, va, k);
    adam4(pb, gb, mb, vb, k);
    __stcs(p4 + i, pa); __stcs(p4 + i + stride, pb);
    __stcs(m4 + i, ma); __stcs(m4 + i + stride, mb);
    __stcs(v4 + i, va); __stcs(v4 + i + stride, vb);
  }
  for (; i < n4; i += stride) {
    float4 pa = __ldcs(p4 + i);
    const float4 ga = __ldcs(g4 + i);
    float4 ma = __ldcs(m4 + i), va = __ldcs(v4 + i);
    adam4(pa, ga, ma, va, k);
    __stcs(p4 + i, pa); __stcs(m4 + i, ma); __stcs(v4 + i, va);
  }
  // ragged tail (< 4 elements)
  const int64_t j = (n4 << 2) + (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (j < n) {
    float pv = p[j], mv = m[j], vv = v[j];
    adam1(pv, g[j], mv, vv, k);
    p[j] = pv; m[j] = mv; v[j] = vv;
  }
}

}  // namespace

cudaError_t launch_adamw(float* p, const float* g, float* m, float* v, int64_t n, const AdamScalars& k,
                         cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int64_t n4 = n >> 2;
  const int64_t want = (n4 + 2 * 256 - 1) / (2 * 256);       // two float4 groups per thread
  int64_t blocks = std::min<int64_t>(want, (int64_t)sms * 8);  // 8 resident CTAs of 256 per SM
  if (blocks < 1) blocks = 1;
  adamw_kernel<<<(unsigned)blocks, 256, 0, s>>>(p, g, m, v, n, k);
  return cudaGetLastError();
}

}  // namespace mfsdp
