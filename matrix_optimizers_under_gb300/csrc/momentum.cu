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
// stored matrix transposed when rows > cols).  A thread holds two runs of 8
// consecutive elements of one stored row, and the 32 lanes of a warp hold 4
// whole stored rows of the tile: every access of a warp -- 16-byte gradient
// loads, 32-byte momentum loads and stores -- covers whole 32-byte sectors
// (4 x 128 bytes of bf16 G, 4 x 256 bytes of M).  Handing each lane 16
// elements of a row instead, with its 16-byte accesses 32 or 64 bytes apart,
// left every sector half used by each access; the L2 then served twice the
// requests, and the phase reached ~78 % of HBM inside the step (after
// Newton-Schulz, at the power-capped clock) against ~95 % now.  Every thread
// issues all its loads before using any, writes M back, and writes
// X0 = bf16(U) into the workspace's blocked, pre-swizzled layout: a run is
// one 16-byte chunk of an atom row when X0 has the stored orientation; for the
// transpose, the tile's X0 block (64 X0 rows = one column block, 8 atoms) is
// assembled in shared memory -- 2-byte stores in an XOR-swizzled image that
// keeps them free of bank conflicts -- and, after one block barrier, each
// warp copies one whole atom out with 16-byte accesses.
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

// Tiles per CTA of the momentum kernel.  Two (every load of both issued
// first, 96 registers, two CTAs per SM) measured 4-17 % slower than one (60
// registers, four CTAs per SM).
constexpr int kMomTilesPerCta = 1;

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Global accesses of the momentum kernel, as volatile asm so that they stay in
// program order (every load of a CTA's tiles is issued before the first
// store).  16-byte and 32-byte (sm_100 and later) vectors, streaming.
__device__ __forceinline__ uint4 ld_cs_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.cs.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ void ld_cs_v8(const void* p, uint32_t (&v)[8]) {
  asm volatile("ld.global.cs.v8.u32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
               : "l"(p));
}
__device__ __forceinline__ void st_cs_v4(void* p, const float* v) {
  asm volatile("st.global.cs.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3])
               : "memory");
}
__device__ __forceinline__ void st_cs_v8(void* p, const float* v) {
  asm volatile("st.global.cs.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "f"(v[0]), "f"(v[1]),
               "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7])
               : "memory");
}

// One thread's share of one tile: 8 consecutive stored elements of one
// stored row (a "run").  Thread t of the CTA holds runs t and t + 256 of the
// tile's 512: run k is stored row r0 + k / 8, stored columns c0 + 8 (k % 8)
// .. + 7.  So the 32 lanes of a warp cover 4 whole stored rows of the tile per
// access: 4 x 128 bytes of a bf16 gradient, 4 x 256 bytes of momentum -- every
// 32-byte sector an access touches is used in full.
constexpr int kRunsPerThread = 2;

struct Run {
  int64_t e;       // stored element index of the run's first element (within the matrix)
  int kind;        // 0: outside the matrix (zeros), 1: vectors, 2: scalar (ragged edge or offset)
  uint32_t g[8];   // bf16 gradient: g[0..3] (8 values); fp32 gradient: g[0..7]
  uint32_t m[8];   // fp32 momentum
};

template <bool kBf16>
__device__ __forceinline__ void issue_run(const MomMat& d, Run& r) {
  if (r.kind != 1) return;
  if constexpr (kBf16) {
    const uint4 q = ld_cs_v4(static_cast<const uint16_t*>(d.g) + r.e);
    r.g[0] = q.x; r.g[1] = q.y; r.g[2] = q.z; r.g[3] = q.w;
  } else {
    const float* gp = static_cast<const float*>(d.g) + r.e;
    if (d.g32) {
      ld_cs_v8(gp, r.g);
    } else {
      const uint4 a = ld_cs_v4(gp), b = ld_cs_v4(gp + 4);
      r.g[0] = a.x; r.g[1] = a.y; r.g[2] = a.z; r.g[3] = a.w; r.g[4] = b.x; r.g[5] = b.y; r.g[6] = b.z; r.g[7] = b.w;
    }
  }
  const float* mp = d.m + r.e;
  if (d.m32) {
    ld_cs_v8(mp, r.m);
  } else {
    const uint4 a = ld_cs_v4(mp), b = ld_cs_v4(mp + 4);
    r.m[0] = a.x; r.m[1] = a.y; r.m[2] = a.z; r.m[3] = a.w; r.m[4] = b.x; r.m[5] = b.y; r.m[6] = b.z; r.m[7] = b.w;
  }
}

template <bool kBf16>
__device__ __forceinline__ float run_g(const Run& r, int e) {
  if constexpr (kBf16) return bf16_bits_to_float((e & 1) ? (r.g[e >> 1] >> 16) : (r.g[e >> 1] & 0xFFFFu));
  return __uint_as_float(r.g[e]);
}

// Momentum of one run: M <- beta M + G written back, u = the Newton-Schulz
// input (M, or G + beta M with nesterov).
template <bool kBf16>
__device__ __forceinline__ void momentum_run(const MomBatch& p, const MomMat& d, const Run& r, int64_t gc,
                                             float (&u)[8]) {
  const float beta = p.beta;
  if (r.kind == 1) {
    float mn[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float g = run_g<kBf16>(r, e);
      mn[e] = fmaf(beta, __uint_as_float(r.m[e]), g);
      u[e] = p.nesterov ? fmaf(beta, mn[e], g) : mn[e];
    }
    float* mp = d.m + r.e;
    if (d.m32) {
      st_cs_v8(mp, mn);
    } else {
      st_cs_v4(mp, mn);
      st_cs_v4(mp + 4, mn + 4);
    }
  } else if (r.kind == 2) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      u[e] = 0.f;
      if (gc + e < d.cols) {
        const int64_t idx = r.e + e;
        const float gv = kBf16 ? bf16_bits_to_float(static_cast<const uint16_t*>(d.g)[idx])
                               : static_cast<const float*>(d.g)[idx];
        const float mnv = fmaf(beta, d.m[idx], gv);
        d.m[idx] = mnv;
        u[e] = p.nesterov ? fmaf(beta, mnv, gv) : mnv;
      }
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) u[e] = 0.f;
  }
}

// Position (in 16-byte chunks) of X0 chunk q of row i (tile-relative) in the
// transpose image: the atom swizzle q ^ (i % 8), further XORed with i / 8.
// A thread's 2-byte stores of one instruction (one value of its run: rows
// 8a + e for a = 0..7, columns four apart per 8 lanes) then hit 8 distinct
// chunk slots of 8 rows, all 32 banks; the copy-out of one atom row group
// reads 4 whole 128-byte image rows per instruction.
__device__ __forceinline__ int xpose_slot(int i, int q) { return (q ^ (i & 7) ^ (i >> 3)) & 7; }

// kTilesPerCta consecutive 64 x 64 tiles of X0 per CTA.  Each thread issues
// every load of its runs in all of them before it uses any, then writes M
// back and X0 = bf16(U) into the workspace's blocked, pre-swizzled layout:
// for X0 in the stored orientation a run is one 16-byte chunk of an atom row
// (the warp writes 512 contiguous bytes of one atom); for the transpose, the
// tile is assembled in shared memory and each warp copies one whole 1 KB atom
// out.  One norm partial per warp and tile (fixed shuffle order).
template <bool kBf16, int kTilesPerCta>
__global__ void __launch_bounds__(256) momentum_kernel(const __grid_constant__ MomBatch p, int total_tiles) {
  __shared__ __align__(16) uint8_t xpose[kTilesPerCta][kTile * kTile * 2];
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int first = blockIdx.x * kTilesPerCta;
  int mi[kTilesPerCta], local[kTilesPerCta];
  Run run[kTilesPerCta][kRunsPerThread];
  int m = find_mat(p.tile_start, p.n, first);
#pragma unroll
  for (int k = 0; k < kTilesPerCta; ++k) {
    const int tile = first + k;
    if (tile < total_tiles) {
      while (m + 1 < p.n && p.tile_start[m + 1] <= tile) ++m;
    }
    mi[k] = m;
    const MomMat& d = p.mat[m];
    local[k] = tile - p.tile_start[m];
    const int ti = local[k] / d.tiles_j, tj = local[k] - ti * d.tiles_j;
    const int64_t r0 = d.transposed ? tj * kTile : ti * kTile;   // stored block of this X0 tile
    const int64_t c0 = d.transposed ? ti * kTile : tj * kTile;
#pragma unroll
    for (int h = 0; h < kRunsPerThread; ++h) {
      Run& r = run[k][h];
      const int64_t gr = r0 + (t >> 3) + 32 * h, gc = c0 + 8 * (t & 7);
      r.e = gr * d.cols + gc;
      r.kind = (tile < total_tiles && gr < d.rows && gc < d.cols) ? ((d.vec_ok && gc + 8 <= d.cols) ? 1 : 2) : 0;
      issue_run<kBf16>(d, r);
    }
  }
  bool any_xpose = false;
#pragma unroll
  for (int k = 0; k < kTilesPerCta; ++k) {
    if (first + k >= total_tiles) break;
    const MomMat& d = p.mat[mi[k]];
    const int ti = local[k] / d.tiles_j, tj = local[k] - ti * d.tiles_j;
    const int i0 = ti * kTile, j0 = tj * kTile;
    float ss = 0.f;
#pragma unroll
    for (int h = 0; h < kRunsPerThread; ++h) {
      const int row = (t >> 3) + 32 * h, col = 8 * (t & 7);       // tile-relative stored row / column
      float u[8];
      momentum_run<kBf16>(p, d, run[k][h], (d.transposed ? i0 : j0) + col, u);
      uint32_t pk[4];
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(u[e], u[e], ss);
#pragma unroll
      for (int q = 0; q < 4; ++q) pk[q] = pack_bf16x2(u[2 * q], u[2 * q + 1]);
      if (!d.transposed) {
        *reinterpret_cast<uint4*>(d.y + blocked_chunk(d.s_pad, i0 + row, j0 + col)) =
            make_uint4(pk[0], pk[1], pk[2], pk[3]);
      } else {
        // X0 rows col .. col+7 (tile-relative) at X0 column row.
        uint16_t* img = reinterpret_cast<uint16_t*>(xpose[k]);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int i = col + e;
          img[i * 64 + xpose_slot(i, row >> 3) * 8 + (row & 7)] =
              (uint16_t)((e & 1) ? (pk[e >> 1] >> 16) : (pk[e >> 1] & 0xFFFFu));
        }
        any_xpose = true;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) p.partials[(size_t)(d.partial0 + local[k]) * 8 + warp] = ss;
  }
  if (__syncthreads_or(any_xpose)) {
    // Warp w writes atom w of each transposed tile's block (X0 rows i0 + 8w ..
    // +7): lane l the 16-byte chunks at positions l and l + 32 of the atom, in
    // the atom's own swizzled order.
#pragma unroll
    for (int k = 0; k < kTilesPerCta; ++k) {
      if (first + k >= total_tiles) break;
      const MomMat& d = p.mat[mi[k]];
      if (!d.transposed) continue;
      const int ti = local[k] / d.tiles_j, tj = local[k] - ti * d.tiles_j;
      const int i0 = ti * kTile, j0 = tj * kTile;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int pos = lane + 32 * h;                 // chunk position within the 1 KB atom
        const int rr = pos >> 3, phys = pos & 7;       // atom row, stored chunk position
        const int i = 8 * warp + rr;                   // X0 row within the tile
        const int q = phys ^ rr;                       // logical chunk (X0 columns 8q .. 8q+7)
        const uint4 v = *reinterpret_cast<const uint4*>(xpose[k] + (i * 64 + xpose_slot(i, q) * 8) * 2);
        *reinterpret_cast<uint4*>(d.y + blocked_chunk(d.s_pad, i0 + i, j0 + 8 * q)) = v;
      }
    }
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
  constexpr int kT = kMomTilesPerCta;
  const int blocks = (total_tiles + kT - 1) / kT;
  if (b.grad_bf16) momentum_kernel<true, kT><<<blocks, 256, 0, s>>>(b, total_tiles);
  else momentum_kernel<false, kT><<<blocks, 256, 0, s>>>(b, total_tiles);
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
