// Segment view + Muon momentum + Frobenius-norm partials (one pass over HBM),
// the deterministic norm finalise, and the emit kernel for zero Newton-Schulz
// steps.
//
// MatrixFSDP: Communication-Free Matrix Optimizers Under ZeRO-3 Parameter
// Sharding -- Abstract: the owner reads each matrix's full reduced gradient
// out of its owner shard through MatrixShard metadata and applies Muon, which
// orthogonalises momentum-smoothed updates.  Readings: heavy-ball momentum
// M <- beta*M + G (U = M, or G + beta*M with nesterov) and the prescale
// X0 = U / (||U||_F + eps) that Newton-Schulz needs.
//
// Each CTA takes one 64 x 64 tile of the Newton-Schulz iterate X0 (s x l, the
// stored matrix transposed when rows > cols).  It reads the matching stored
// block of G and M once (16-byte vectors when the segment allows), writes M
// back, stages U in shared memory, and writes X0 = bf16(U) as eight 1 KB
// pre-swizzled atoms of the workspace's blocked layout -- transposing through
// shared memory for tall matrices, so every later GEMM sees the short side
// first.  The padding up to multiples of 128 is written as zeros.  The per-CTA
// sum of U^2 (fp32, warp shuffles then a fixed-order block sum) goes to its own
// slot; the finalise kernel adds a matrix's slots in a fixed order, so the
// norm is bitwise reproducible.  HBM traffic: 2 (bf16 G) + 4 + 4 (M) + 2 (X0)
// = 12 bytes per element.
#include <cuda_bf16.h>

#include "mfsdp_internal.h"

namespace mfsdp {
namespace {

__device__ __forceinline__ int find_mat(const int32_t* start, int n, int t) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (start[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__global__ void __launch_bounds__(256) momentum_kernel(const __grid_constant__ MomBatch p) {
  __shared__ float tile[kTile][kTile + 1];
  __shared__ float warp_sum[8];
  const int t = threadIdx.x;
  const int mi = find_mat(p.tile_start, p.n, blockIdx.x);
  const MomMat& d = p.mat[mi];
  const int local = blockIdx.x - p.tile_start[mi];
  const int ti = local / d.tiles_j, tj = local - ti * d.tiles_j;
  const int i0 = ti * kTile, j0 = tj * kTile;       // tile origin in X0 (s x l)
  const int64_t r0 = d.transposed ? j0 : i0;         // matching stored block
  const int64_t c0 = d.transposed ? i0 : j0;

  const int lr = t >> 2, lc = (t & 3) * 16;
  const int64_t gr = r0 + lr, gc = c0 + lc;
  const float beta = p.beta;
  float u[16];
  float ss = 0.f;
  if (gr < d.rows && gc < d.cols) {
    const int64_t e0 = gr * d.cols + gc;
    if (d.vec_ok && gc + 16 <= d.cols) {
      float g[16];
      if (p.grad_bf16) {
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(d.g) + e0);
        const uint4 q0 = __ldcs(src), q1 = __ldcs(src + 1);
        const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          g[2 * k] = bf16_bits_to_float(w[k] & 0xFFFFu);
          g[2 * k + 1] = bf16_bits_to_float(w[k] >> 16);
        }
      } else {
        const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(d.g) + e0);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float4 q = __ldcs(src + k);
          g[4 * k] = q.x; g[4 * k + 1] = q.y; g[4 * k + 2] = q.z; g[4 * k + 3] = q.w;
        }
      }
      float4* mp = reinterpret_cast<float4*>(d.m + e0);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float4 q = __ldcs(mp + k);
        float mv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float gv = g[4 * k + e];
          const float mn = fmaf(beta, mv[e], gv);
          mv[e] = mn;
          u[4 * k + e] = p.nesterov ? fmaf(beta, mn, gv) : mn;
        }
        __stcs(mp + k, make_float4(mv[0], mv[1], mv[2], mv[3]));
      }
    } else {
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        u[e] = 0.f;
        if (gc + e < d.cols) {
          const int64_t idx = e0 + e;
          const float gv = p.grad_bf16 ? bf16_bits_to_float(static_cast<const uint16_t*>(d.g)[idx])
                                       : static_cast<const float*>(d.g)[idx];
          const float mn = fmaf(beta, d.m[idx], gv);
          d.m[idx] = mn;
          u[e] = p.nesterov ? fmaf(beta, mn, gv) : mn;
        }
      }
    }
  } else {
#pragma unroll
    for (int e = 0; e < 16; ++e) u[e] = 0.f;
  }
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    ss = fmaf(u[e], u[e], ss);
    tile[lr][lc + e] = u[e];
  }
  __syncthreads();

  // X0 tile rows [i0, i0+64), columns [j0, j0+64): 64 rows x 8 chunks of 8.
  const size_t stride = colblock_stride(d.s_pad);
#pragma unroll
  for (int it = 0; it < 2; ++it) {
    const int q = t + 256 * it;
    const int yi = q >> 3, ch = q & 7;
    float v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = d.transposed ? tile[ch * 8 + e][yi] : tile[yi][ch * 8 + e];
    uint4 w;
    w.x = pack_bf16x2(v[0], v[1]);
    w.y = pack_bf16x2(v[2], v[3]);
    w.z = pack_bf16x2(v[4], v[5]);
    w.w = pack_bf16x2(v[6], v[7]);
    const int row = i0 + yi;
    uint8_t* dst = d.y + (size_t)(j0 >> 6) * stride + (size_t)(row >> 3) * 1024 + (size_t)(row & 7) * 128 +
                   (size_t)((ch ^ (row & 7)) << 4);
    *reinterpret_cast<uint4*>(dst) = w;
  }

  // Fixed-order reduction of the tile's sum of squares.
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((t & 31) == 0) warp_sum[t >> 5] = ss;
  __syncthreads();
  if (t == 0) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) s += warp_sum[w];
    p.partials[d.partial0 + local] = s;
  }
}

__global__ void __launch_bounds__(256) norm_finalize_kernel(const __grid_constant__ NormBatch p) {
  __shared__ float warp_sum[8];
  const int i = blockIdx.x;
  const int b = p.start[i], e = p.start[i + 1];
  float s = 0.f;
  for (int k = b + (int)threadIdx.x; k < e; k += 256) s += p.partials[k];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) warp_sum[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) tot += warp_sum[w];
    p.norm[p.first + i] = make_float2(tot, 1.0f / (sqrtf(tot) + p.eps));
  }
}

// Zero Newton-Schulz steps: update = X0 / (||U|| + eps), in the stored layout.
__global__ void __launch_bounds__(256) emit_kernel(const __grid_constant__ EmitBatch p) {
  const int mi = find_mat(p.tile_start, p.n, blockIdx.x);
  const EmitMat& d = p.mat[mi];
  const int local = blockIdx.x - p.tile_start[mi];
  const int ti = local / d.tiles_j, tj = local - ti * d.tiles_j;
  const float2 nrm = p.norm[d.norm_idx];
  const float scale = nrm.x == 0.f ? 0.f : nrm.y;
  for (int e = threadIdx.x; e < kTile * kTile; e += 256) {
    // consecutive threads walk the stored matrix's contiguous dimension
    const int a = e & (kTile - 1), bb = e >> 6;
    const int yi = ti * kTile + (d.transposed ? a : bb);   // X0 row (short side)
    const int yj = tj * kTile + (d.transposed ? bb : a);   // X0 column (long side)
    const int64_t sr = d.transposed ? yj : yi, sc = d.transposed ? yi : yj;
    if (sr >= d.rows || sc >= d.cols) continue;
    const uint16_t bits =
        *reinterpret_cast<const uint16_t*>(d.y + blocked_chunk(d.s_pad, yi, yj & ~7) + (size_t)(yj & 7) * 2);
    const float v = bf16_bits_to_float(bits) * scale;
    const int64_t o = sr * d.cols + sc;
    if (p.out_bf16) static_cast<__nv_bfloat16*>(d.out)[o] = __float2bfloat16_rn(v);
    else static_cast<float*>(d.out)[o] = v;
  }
}

}  // namespace

cudaError_t launch_momentum(const MomBatch& b, int total_tiles, cudaStream_t s) {
  if (total_tiles <= 0) return cudaSuccess;
  momentum_kernel<<<total_tiles, 256, 0, s>>>(b);
  return cudaGetLastError();
}

cudaError_t launch_norm_finalize(const NormBatch& b, cudaStream_t s) {
  if (b.n <= 0) return cudaSuccess;
  norm_finalize_kernel<<<b.n, 256, 0, s>>>(b);
  return cudaGetLastError();
}

cudaError_t launch_emit(const EmitBatch& b, int total_tiles, cudaStream_t s) {
  if (total_tiles <= 0) return cudaSuccess;
  emit_kernel<<<total_tiles, 256, 0, s>>>(b);
  return cudaGetLastError();
}

}  // namespace mfsdp
