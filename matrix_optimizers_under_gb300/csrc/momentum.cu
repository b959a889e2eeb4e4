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
// stored matrix transposed when rows > cols).  Every thread issues all its
// loads of the matching stored G and M (16-byte vectors when the segment
// allows) before using any, writes M back, and writes X0 = bf16(U) into the
// workspace's blocked, pre-swizzled layout: straight from registers when X0
// has the stored orientation (each warp fills one 1 KB atom).  When X0 is the
// transpose, the tile's X0 block (64 X0 rows = one column block, 8 atoms) is
// assembled in shared memory -- 2-byte stores in an XOR-swizzled image that
// keeps them free of bank conflicts -- and, after one block barrier, each warp
// copies one whole atom out with 16-byte accesses, so every X0 line is written
// in full by one warp (writing 16-byte pieces of 64 different lines per warp
// held tall matrices to ~72 % of HBM against ~88 % for wide ones).
// The padding up to multiples of 128 is written as zeros.  Each warp's sum of
// U^2 (fp32, fixed shuffle order) goes to its own slot; the finalise kernel
// adds a matrix's slots in a fixed order, so the norm is bitwise
// reproducible.  HBM traffic: 2 (bf16 G) + 4 + 4 (M) + 2 (X0) = 12 bytes per
// element.
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

// 16 consecutive elements of one stored row: gradient as fp32, momentum.
struct Row16 {
  float g[16];
  float m[16];
};

__device__ __forceinline__ void load_row16_vec(const MomMat& d, int grad_bf16, int64_t e0, Row16& r) {
  // All six (bf16) or eight (fp32) 16-byte loads are issued before any use.
  const float4* mp = reinterpret_cast<const float4*>(d.m + e0);
  float4 mq[4];
  if (grad_bf16) {
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(d.g) + e0);
    const uint4 q0 = __ldcs(src), q1 = __ldcs(src + 1);
#pragma unroll
    for (int k = 0; k < 4; ++k) mq[k] = __ldcs(mp + k);
    const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      r.g[2 * k] = bf16_bits_to_float(w[k] & 0xFFFFu);
      r.g[2 * k + 1] = bf16_bits_to_float(w[k] >> 16);
    }
  } else {
    const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(d.g) + e0);
    float4 gq[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) gq[k] = __ldcs(src + k);
#pragma unroll
    for (int k = 0; k < 4; ++k) mq[k] = __ldcs(mp + k);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      r.g[4 * k] = gq[k].x; r.g[4 * k + 1] = gq[k].y; r.g[4 * k + 2] = gq[k].z; r.g[4 * k + 3] = gq[k].w;
    }
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    r.m[4 * k] = mq[k].x; r.m[4 * k + 1] = mq[k].y; r.m[4 * k + 2] = mq[k].z; r.m[4 * k + 3] = mq[k].w;
  }
}

// Position (in 16-byte chunks) of chunk q of X0 row i (both within the tile) in
// the transpose buffer: the atom swizzle q ^ (i % 8), further XORed with
// 2 * ((i / 16) % 4) so that the 2-byte stores of one warp instruction -- rows
// 16a + e for a = 0..3, one chunk, eight row pairs -- fall in 16 distinct banks.
__device__ __forceinline__ int xpose_slot(int i, int q) { return (q ^ (i & 7) ^ (((i >> 4) & 3) << 1)) & 7; }

// One CTA = one 64 x 64 tile of X0; warp w owns stored rows [r0 + 8w, r0 + 8w + 8),
// lane l row r0 + 8w + l/4 and stored columns [c0 + 16(l%4), +16).  Every warp
// writes its own norm partial.
__global__ void __launch_bounds__(256) momentum_kernel(const __grid_constant__ MomBatch p) {
  __shared__ __align__(16) uint8_t xpose[kTile * kTile * 2];   // transposed tiles: the X0 block, 8 atoms
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int mi = find_mat(p.tile_start, p.n, blockIdx.x);
  const MomMat& d = p.mat[mi];
  const int local = blockIdx.x - p.tile_start[mi];
  const int ti = local / d.tiles_j, tj = local - ti * d.tiles_j;
  const int i0 = ti * kTile, j0 = tj * kTile;       // tile origin in X0 (s x l)
  const int64_t r0 = d.transposed ? j0 : i0;         // matching stored block
  const int64_t c0 = d.transposed ? i0 : j0;

  const int lr = warp * 8 + (lane >> 2), lc = (lane & 3) * 16;
  const int64_t gr = r0 + lr, gc = c0 + lc;
  const float beta = p.beta;
  float u[16];
  float ss = 0.f;
  if (gr < d.rows && gc < d.cols) {
    const int64_t e0 = gr * d.cols + gc;
    if (d.vec_ok && gc + 16 <= d.cols) {
      Row16 r;
      load_row16_vec(d, p.grad_bf16, e0, r);
      float mn[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        mn[e] = fmaf(beta, r.m[e], r.g[e]);
        u[e] = p.nesterov ? fmaf(beta, mn[e], r.g[e]) : mn[e];
      }
      float4* mp = reinterpret_cast<float4*>(d.m + e0);
#pragma unroll
      for (int k = 0; k < 4; ++k) __stcs(mp + k, make_float4(mn[4 * k], mn[4 * k + 1], mn[4 * k + 2], mn[4 * k + 3]));
    } else {
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        u[e] = 0.f;
        if (gc + e < d.cols) {
          const int64_t idx = e0 + e;
          const float gv = p.grad_bf16 ? bf16_bits_to_float(static_cast<const uint16_t*>(d.g)[idx])
                                       : static_cast<const float*>(d.g)[idx];
          const float mnv = fmaf(beta, d.m[idx], gv);
          d.m[idx] = mnv;
          u[e] = p.nesterov ? fmaf(beta, mnv, gv) : mnv;
        }
      }
    }
  } else {
#pragma unroll
    for (int e = 0; e < 16; ++e) u[e] = 0.f;
  }
#pragma unroll
  for (int e = 0; e < 16; ++e) ss = fmaf(u[e], u[e], ss);
  uint32_t pk[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) pk[k] = pack_bf16x2(u[2 * k], u[2 * k + 1]);

  if (!d.transposed) {
    // X0 row = stored row: two 16-byte chunks straight from registers; the warp
    // writes one whole 1 KB atom (8 rows x 64 columns).
    const int row = i0 + lr;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int col = j0 + lc + 8 * h;
      uint8_t* dst = d.y + blocked_chunk(d.s_pad, row, col);
      *reinterpret_cast<uint4*>(dst) = make_uint4(pk[4 * h], pk[4 * h + 1], pk[4 * h + 2], pk[4 * h + 3]);
    }
  } else {
    // X0 row i = stored column i, X0 column j = stored row j.  This thread's
    // 16 values are X0 rows lc .. lc+15 (tile-relative) at X0 column lr:
    // chunk lr / 8 = warp, element lr % 8 of it.
    uint16_t* img = reinterpret_cast<uint16_t*>(xpose);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int i = lc + e;
      const uint32_t word = pk[e >> 1];
      img[i * 64 + xpose_slot(i, warp) * 8 + (lane >> 2)] = (uint16_t)((e & 1) ? (word >> 16) : (word & 0xFFFFu));
    }
    __syncthreads();
    // Warp w writes atom w of the block (X0 rows i0 + 8w .. +7): lane l the
    // 16-byte chunks at positions l and l + 32 of the atom, in the atom's own
    // swizzled order.
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int pos = lane + 32 * h;                 // chunk position within the 1 KB atom
      const int r = pos >> 3, phys = pos & 7;        // atom row, stored chunk position
      const int i = 8 * warp + r;                    // X0 row within the tile
      const int q = phys ^ r;                        // logical chunk (X0 columns 8q .. 8q+7)
      const uint4 v = *reinterpret_cast<const uint4*>(xpose + (i * 64 + xpose_slot(i, q) * 8) * 2);
      *reinterpret_cast<uint4*>(d.y + blocked_chunk(d.s_pad, i0 + i, j0 + 8 * q)) = v;
    }
  }

  // Fixed-order warp reduction; one partial per warp.
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) p.partials[(size_t)(d.partial0 + local) * 8 + warp] = ss;
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
