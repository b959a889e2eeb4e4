// Newton-Schulz products on 5th-generation tensor cores (tcgen05 / TMEM),
// grouped over every matrix of an owner set in one launch per product.
//
// MatrixFSDP: Communication-Free Matrix Optimizers Under ZeRO-3 Parameter
// Sharding -- Abstract: Muon orthogonalises each owned matrix with
// Newton-Schulz locally on its owner.  Muon's quintic iteration on the short
// side (X is s x l):
//     A = X X^T              (kGram,   K = l)
//     B = b A + c A A        (kPoly,   K = s; A is symmetric so A A = A A^T)
//     X <- a X + B X         (kUpdate, K = s)
// with the Frobenius prescale 1/(||U||+eps) folded into the first iteration's
// epilogues (A scaled by its square, the new X by it).
//
// Operands live in the workspace in a blocked layout whose every 1 KB atom
// (8 rows x 64 bf16 columns) is already in the UMMA 128-byte-swizzle order, with
// atoms of one 64-column block contiguous.  So an operand tile of a pipeline
// stage is one contiguous run (or four, for the MN-major X of kUpdate), and a
// 1-D TMA bulk copy (cp.async.bulk) lands it in shared memory ready for
// tcgen05.mma: no tensor maps, any mix of shapes in one launch, and the same
// stored X serves as the K-major operand of the Gram product and the MN-major
// operand of the update.
//
// One CTA computes one 128 x 256 (or 128 x 128) output tile: warp 0 / lane 0
// streams K in 64-element stages through a 4-deep mbarrier ring, warp 1 /
// lane 0 issues 128 x N x 16 UMMAs into a TMEM accumulator, then all four warps
// read the accumulator (tcgen05.ld, one TMEM lane quadrant each), apply the
// fused polynomial epilogue in fp32 and store bf16 (or the final update in the
// caller's dtype and layout, transposed back for tall matrices).  Every wait is
// bounded: on expiry the CTA records kStatusTimeout, drains what it issued,
// frees TMEM and returns.
#include <cuda_bf16.h>

#include "mfsdp_internal.h"
#include "ptx.cuh"

namespace mfsdp {
namespace {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr uint32_t kTmemCols = 256;

__device__ __forceinline__ int find_mat(const int32_t* start, int n, int t) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (start[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Unpack 32 bf16 (four 16-byte chunks) into fp32.
__device__ __forceinline__ void load_bf16x32(const uint8_t* base, const size_t (&off)[4], float (&x)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 w = *reinterpret_cast<const uint4*>(base + off[q]);
    x[8 * q + 0] = bf_lo(w.x); x[8 * q + 1] = bf_hi(w.x);
    x[8 * q + 2] = bf_lo(w.y); x[8 * q + 3] = bf_hi(w.y);
    x[8 * q + 4] = bf_lo(w.z); x[8 * q + 5] = bf_hi(w.z);
    x[8 * q + 6] = bf_lo(w.w); x[8 * q + 7] = bf_hi(w.w);
  }
}

__device__ __forceinline__ void store_bf16x32(uint8_t* base, const size_t (&off)[4], const float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 w;
    w.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
    w.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
    w.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
    w.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
    *reinterpret_cast<uint4*>(base + off[q]) = w;
  }
}

// Final update for 32 consecutive X columns [n, n+32) of X row m, written in
// the caller's layout: stored (m, n) when not transposed, (n, m) otherwise.
__device__ __forceinline__ void store_final(const GemmMat& d, int out_bf16, int m, int n, const float (&v)[32]) {
  if (m >= d.s) return;
  if (!d.transposed) {
    const int64_t row0 = (int64_t)m * d.l;
    if (d.vec_ok && n + 32 <= d.l) {
      if (out_bf16) {
        uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(d.out) + row0 + n);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 w;
          w.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
          w.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
          w.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
          w.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
          o[q] = w;
        }
      } else {
        float4* o = reinterpret_cast<float4*>(static_cast<float*>(d.out) + row0 + n);
#pragma unroll
        for (int q = 0; q < 8; ++q) o[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (n + j < d.l) {
          if (out_bf16) static_cast<__nv_bfloat16*>(d.out)[row0 + n + j] = __float2bfloat16_rn(v[j]);
          else static_cast<float*>(d.out)[row0 + n + j] = v[j];
        }
      }
    }
  } else {
    // stored matrix is l x s: element (n + j, m); the warp's 32 rows m are
    // contiguous in memory, so each j is one coalesced store.
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (n + j < d.l) {
        const int64_t o = (int64_t)(n + j) * d.s + m;
        if (out_bf16) static_cast<__nv_bfloat16*>(d.out)[o] = __float2bfloat16_rn(v[j]);
        else static_cast<float*>(d.out)[o] = v[j];
      }
    }
  }
}

__global__ void __launch_bounds__(kGemmThreads, 1) ns_gemm_kernel(const __grid_constant__ GemmBatch p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ __align__(8) uint64_t done_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mi = find_mat(p.tile_start, p.n, blockIdx.x);
  const GemmMat& d = p.mat[mi];
  const int local = blockIdx.x - p.tile_start[mi];
  const int mt = local % d.tiles_m, nt = local / d.tiles_m;   // m fastest: neighbours share B-operand columns
  const int m0 = mt * kBlockM, n0 = nt * kBlockN;
  const int N = (nt == d.tiles_n - 1) ? d.n_last : kBlockN;
  const int mode = p.mode;

  // A matrix whose momentum is exactly zero has X = 0 throughout: skip the
  // products, and write the zero update once at the end.
  const float2 nrm = p.norm[d.norm_idx];
  if (nrm.x == 0.0f) {
    if (mode == kUpdateFinal) {
      const int m = m0 + threadIdx.x;
      float z[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) z[j] = 0.f;
      for (int c = 0; c < N; c += 32) store_final(d, p.out_bf16, m, n0 + c, z);
    }
    return;
  }

  const uint32_t smem_base = (ptx::smem_u32(smem_raw) + 1023u) & ~1023u;
  auto stage_a = [&](int s) { return smem_base + (uint32_t)s * kStageBytes; };
  auto stage_b = [&](int s) { return smem_base + (uint32_t)s * kStageBytes + kStageBytesA; };

  if (warp == 0) {
    ptx::tmem_alloc(ptx::smem_u32(&tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  if (threadIdx.x == 32) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(ptx::smem_u32(&full_bar[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&empty_bar[s]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&done_bar), 1);
    abort_flag = 0;
    ptx::fence_barrier_init();
    ptx::fence_proxy_async_smem();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_d = tmem_slot;

  const int kb_total = d.k_blocks;
  const size_t a_kstride = colblock_stride(d.s_pad);   // every operand has s_pad rows per column block
  const bool b_mn = (mode == kUpdate || mode == kUpdateFinal);

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      const uint64_t pol = ptx::policy_evict_last();
      const uint32_t a_bytes = kStageBytesA;
      const uint32_t b_bytes = (uint32_t)N * kBlockK * 2;
      int issued = 0;
      for (int kb = 0; kb < kb_total; ++kb) {
        const int s = kb % kStages;
        if (kb >= kStages) {
          if (!ptx::mbar_wait(ptx::smem_u32(&empty_bar[s]), ((kb / kStages) - 1) & 1, kWaitLimitNs)) {
            atomicOr(p.status, kStatusTimeout);
            atomicExch(&abort_flag, 1);
            break;
          }
        }
        if (*(volatile int*)&abort_flag) break;
        const uint32_t fb = ptx::smem_u32(&full_bar[s]);
        ptx::mbar_arrive_expect_tx(fb, a_bytes + b_bytes);
        ptx::bulk_g2s(stage_a(s), d.a_op + (size_t)kb * a_kstride + (size_t)(m0 >> 3) * 1024, a_bytes, fb, pol);
        if (!b_mn) {
          ptx::bulk_g2s(stage_b(s), d.b_op + (size_t)kb * a_kstride + (size_t)(n0 >> 3) * 1024, b_bytes, fb, pol);
        } else {
          // X as the MN-major operand: K rows [64 kb, 64 kb + 64) of column
          // blocks n0/64 ..; each block's 8 atoms are one 8 KB run.
          for (int j = 0; j < N / 64; ++j) {
            const uint8_t* src = d.b_op + (size_t)((n0 >> 6) + j) * a_kstride + (size_t)kb * 8 * 1024;
            ptx::bulk_g2s(stage_b(s) + (uint32_t)j * 8192u, src, 8192u, fb, pol);
          }
        }
        issued = kb + 1;
      }
      // Drain: wait (bounded) until the copies of the last uses of each stage landed.
      for (int kb = (issued > kStages ? issued - kStages : 0); kb < issued; ++kb) {
        ptx::mbar_wait(ptx::smem_u32(&full_bar[kb % kStages]), (kb / kStages) & 1, kWaitLimitNs);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // --------------------------------------------------------- MMA issuer
      const uint32_t idesc = ptx::idesc_bf16_f32(kBlockM, (uint32_t)N, b_mn ? 1u : 0u);
      for (int kb = 0; kb < kb_total; ++kb) {
        const int s = kb % kStages;
        if (!ptx::mbar_wait(ptx::smem_u32(&full_bar[s]), (kb / kStages) & 1, kWaitLimitNs)) {
          atomicOr(p.status, kStatusTimeout);
          atomicExch(&abort_flag, 1);
          break;
        }
        if (*(volatile int*)&abort_flag) break;
        ptx::tc_fence_after();
#pragma unroll
        for (int k = 0; k < kBlockK / 16; ++k) {
          // K-major operand: advance 16 elements (32 bytes) inside the swizzle row.
          const uint64_t adesc = ptx::smem_desc_sw128(stage_a(s) + (uint32_t)k * 32u, 16u, 1024u);
          uint64_t bdesc;
          if (!b_mn) {
            bdesc = ptx::smem_desc_sw128(stage_b(s) + (uint32_t)k * 32u, 16u, 1024u);
          } else {
            // MN-major operand: 16 K rows = two 8-row atoms (2 KB); 64-column
            // blocks 8 KB apart (leading byte offset), 8-row K groups 1 KB
            // apart (stride byte offset).
            bdesc = ptx::smem_desc_sw128(stage_b(s) + (uint32_t)k * 2048u, 8192u, 1024u);
          }
          ptx::umma_bf16(tmem_d, adesc, bdesc, idesc, (kb > 0 || k > 0) ? 1u : 0u);
        }
        ptx::umma_commit(ptx::smem_u32(&empty_bar[s]));   // frees the stage once these MMAs finish
      }
      ptx::umma_commit(ptx::smem_u32(&done_bar));        // accumulator complete (or drained on abort)
    }
    __syncwarp();
  }

  // ------------------------------------------------------------------ epilogue
  const bool done_ok = ptx::mbar_wait(ptx::smem_u32(&done_bar), 0, kWaitLimitNs);
  if (!done_ok) {
    if (lane == 0) atomicOr(p.status, kStatusTimeout);
    atomicExch(&abort_flag, 1);
  }
  ptx::tc_fence_after();
  __syncwarp();
  const bool write = done_ok && !*(volatile int*)&abort_flag;
  if (done_ok) {
    const int m = m0 + warp * 32 + lane;                         // this thread's output row
    const uint32_t t_row = tmem_d + ((uint32_t)(warp * 32) << 16);
    const float scale_gram = p.first_iter ? nrm.y * nrm.y : 1.0f;
    const float scale_upd = p.first_iter ? nrm.y : 1.0f;
    const size_t stride = colblock_stride(d.s_pad);
    const size_t row_off = (size_t)(m >> 3) * 1024 + (size_t)(m & 7) * 128;
    for (int c = 0; c < N; c += 32) {
      uint32_t r[32];
      ptx::tmem_ld_32x32b_x32(t_row + (uint32_t)c, r);
      ptx::tmem_ld_wait();
      if (!write) continue;
      const int n = n0 + c;
      size_t off[4];
      const size_t base = (size_t)(n >> 6) * stride + row_off;
#pragma unroll
      for (int q = 0; q < 4; ++q) off[q] = base + (size_t)(((((n & 63) >> 3) + q) ^ (m & 7)) << 4);
      float v[32];
      if (mode == kGram) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]) * scale_gram;
        store_bf16x32(static_cast<uint8_t*>(d.out), off, v);
      } else if (mode == kPoly) {
        float x[32];
        load_bf16x32(d.c_in, off, x);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = fmaf(p.c, __uint_as_float(r[j]), p.b * x[j]);
        store_bf16x32(static_cast<uint8_t*>(d.out), off, v);
      } else {
        float x[32];
        load_bf16x32(d.c_in, off, x);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = fmaf(p.a, x[j], __uint_as_float(r[j])) * scale_upd;
        if (mode == kUpdate) store_bf16x32(static_cast<uint8_t*>(d.out), off, v);
        else store_final(d, p.out_bf16, m, n, v);
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_d, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_ns_gemm(const GemmBatch& b, int total_tiles, cudaStream_t s) {
  if (total_tiles <= 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(ns_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kGemmSmemBytes);
  if (e != cudaSuccess) return e;
  ns_gemm_kernel<<<total_tiles, kGemmThreads, kGemmSmemBytes, s>>>(b);
  return cudaGetLastError();
}

}  // namespace mfsdp
