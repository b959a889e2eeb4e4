// Owner-segment reduce and owner-shard resharding: one HBM-bound kernel that
// moves (and optionally sums) element segments between flat buffers.
//
// MatrixFSDP: Communication-Free Matrix Optimizers Under ZeRO-3 Parameter
// Sharding -- Abstract: the ordinary backward reduction lands each matrix's full
// gradient on its owner -- an uneven reduce-scatter over owner segments, made
// deterministic by owner-segment collectives -- and owner-shard checkpoint
// resharding moves owner-shaped shards between layouts.  FAQ (docshare page):
// owner segments replace equal-size shard assumptions.
//
// On one GPU the data-parallel ranks are simulated: their local gradients are
// separate flat buffers.  REDUCE sums, for every segment, all sources in rank
// order in fp32 and rounds once to the destination dtype, so the result is
// bitwise reproducible; GATHER copies each segment from its own source.  A CTA
// takes a chunk of 2048 elements of one segment; each thread moves 8
// consecutive elements, with 16-byte vectors when both ends allow it.
#include <cuda_bf16.h>

#include "mfsdp_internal.h"

namespace mfsdp {
namespace {

__device__ __forceinline__ int find_seg(const int32_t* start, int n, int t) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (start[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ float load_elem(const void* base, int64_t i, int bf16) {
  return bf16 ? __uint_as_float((uint32_t)static_cast<const uint16_t*>(base)[i] << 16)
              : static_cast<const float*>(base)[i];
}

// 8 consecutive elements; 16-byte loads when `vec`, else element by element
// with the ones at or beyond `cnt` read as zero.
__device__ __forceinline__ void load8(const void* base, int64_t i, int bf16, bool vec, int cnt, float (&x)[8]) {
  if (vec) {
    if (bf16) {
      const uint4 q = __ldcs(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + i));
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        x[2 * k] = __uint_as_float(w[k] << 16);
        x[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
      }
    } else {
      const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + i);
      const float4 a = __ldcs(p), b = __ldcs(p + 1);
      x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = k < cnt ? load_elem(base, i + k, bf16) : 0.f;
  }
}

__global__ void __launch_bounds__(256) segment_kernel(const __grid_constant__ SegBatch p) {
  const int si = find_seg(p.chunk_start, p.n, blockIdx.x);
  const SegDesc& g = p.seg[si];
  const int64_t e0 = (int64_t)(blockIdx.x - p.chunk_start[si]) * kSegChunk + (int64_t)threadIdx.x * 8;
  if (e0 >= g.numel) return;
  const int64_t rem = g.numel - e0;
  const int cnt = rem < 8 ? (int)rem : 8;
  const int64_t s0 = g.src_offset + e0, d0 = g.dst_offset + e0;
  const bool vin = cnt == 8 && (s0 & 7) == 0;     // every base pointer is 16-byte aligned
  const bool vout = cnt == 8 && (d0 & 7) == 0;
  float acc[8];
  if (p.mode == 0) {
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = 0.f;
    for (int r = 0; r < p.n_src; ++r) {             // rank order: bitwise reproducible
      float x[8];
      load8(p.src[r], s0, p.src_bf16, vin, cnt, x);
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[k] += x[k];
    }
  } else {
    load8(p.src[g.src_index], s0, p.src_bf16, vin, cnt, acc);
  }
  if (p.dst_bf16) {
    __nv_bfloat16* d = static_cast<__nv_bfloat16*>(p.dst) + d0;
    if (vout) {
      __nv_bfloat162 h[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) h[k] = __floats2bfloat162_rn(acc[2 * k], acc[2 * k + 1]);
      __stcs(reinterpret_cast<uint4*>(d), *reinterpret_cast<const uint4*>(h));
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (k < cnt) d[k] = __float2bfloat16_rn(acc[k]);
    }
  } else {
    float* d = static_cast<float*>(p.dst) + d0;
    if (vout) {
      __stcs(reinterpret_cast<float4*>(d), make_float4(acc[0], acc[1], acc[2], acc[3]));
      __stcs(reinterpret_cast<float4*>(d) + 1, make_float4(acc[4], acc[5], acc[6], acc[7]));
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (k < cnt) d[k] = acc[k];
    }
  }
}

}  // namespace

cudaError_t launch_segments(const SegBatch& b, int total_chunks, cudaStream_t s) {
  if (total_chunks <= 0) return cudaSuccess;
  segment_kernel<<<total_chunks, 256, 0, s>>>(b);
  return cudaGetLastError();
}

}  // namespace mfsdp
