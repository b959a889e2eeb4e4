// Launch descriptors shared by the host orchestration (host.cu) and the
// kernels.  Every launch carries its per-matrix table by value as a
// __grid_constant__ kernel parameter, so a step needs no device-side metadata
// upload and can be captured in a CUDA graph as plain kernel nodes.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "mfsdp.h"

namespace mfsdp {

constexpr int kMaxBatch = 128;     // matrices per launch
constexpr int kTile = 64;          // momentum-kernel tile edge (elements)
constexpr int kPartialsPerTile = 8;  // momentum kernel: one norm partial per warp
constexpr int kPad = 128;          // workspace: the long side is padded to a multiple of this
constexpr int kPadS = 256;         // workspace: the short side is padded to a multiple of this (one CTA pair)
constexpr int kBlockM = 128;       // Newton-Schulz GEMM tile rows per CTA (its TMEM lanes)
constexpr int kPairM = 2 * kBlockM;  // rows of the tile a CTA pair computes (pair UMMA, M = 256)
constexpr int kBlockN = 256;       // Newton-Schulz GEMM tile columns (UMMA N)
constexpr int kAtomK = 64;         // K elements of one 128-byte swizzle row (a column block of the layout)
constexpr int kBlockK = 128;       // K elements per pipeline stage: two column blocks
constexpr int kStages = 3;         // smem pipeline depth
constexpr int kStageBytesA = kBlockM * kBlockK * 2;         // 32 KB: this CTA's 128 rows of A
constexpr int kStageBytesB = (kBlockN / 2) * kBlockK * 2;   // 32 KB: this CTA's half of B's columns
constexpr int kStageBytes = kStageBytesA + kStageBytesB;
constexpr int kEpilogueWarps = 8;  // warps 2-9 of the GEMM CTA: two per TMEM lane quadrant
constexpr int kSchedulerWarp = 2 + kEpilogueWarps;        // warp 10: hands out ready tiles
constexpr int kGemmThreads = 32 * (kSchedulerWarp + 1);   // producer, MMA, epilogue warps, scheduler
constexpr int kStageOutBytes = kBlockM * kAtomK * 2;   // 16 KB: one 128-row x 64-column block of the epilogue
// the stages, one epilogue staging block per half of the epilogue warps, alignment slack
constexpr size_t kGemmSmemBytes = (size_t)kStages * kStageBytes + 2 * (size_t)kStageOutBytes + 1024;

// Bytes between consecutive 64-column blocks of a blocked matrix with rows_pad rows.
__host__ __device__ inline size_t colblock_stride(int rows_pad) { return (size_t)rows_pad * 128; }

// Byte offset of the 16-byte chunk holding columns [col, col+8) of row `row`
// (col a multiple of 8) in the blocked, pre-swizzled layout: 1024-byte atoms of
// 8 rows x 64 bf16 columns, atoms column-block major, chunk index XOR row%8 --
// the exact image of the UMMA 128-byte-swizzle canonical layout.
__host__ __device__ inline size_t blocked_chunk(int rows_pad, int row, int col) {
  return (size_t)(col >> 6) * colblock_stride(rows_pad) + (size_t)(row >> 3) * 1024 +
         (size_t)(row & 7) * 128 + (size_t)((((col & 63) >> 3) ^ (row & 7)) << 4);
}

// ---------------------------------------------------------------- momentum (K1)
struct MomMat {
  const void* g;       // gradient at the shard's offset (fp32 or bf16)
  float* m;            // momentum at the shard's offset
  uint8_t* y;          // X0 in the workspace (blocked bf16, s_pad x l_pad)
  int64_t rows, cols;  // stored shape
  int32_t s_pad, l_pad;
  int32_t transposed;
  int32_t vec_ok;      // offset and cols multiples of 8: every run of 8 elements of a row is a vector
  int32_t g32, m32;    // the matrix's first gradient / momentum element is 32-byte aligned (256-bit access)
  int32_t tiles_j;     // l_pad / kTile
  int32_t partial0;    // first tile index of this matrix (its partial slots start at 8x this)
};
struct MomBatch {
  int32_t n;
  int32_t grad_bf16;
  int32_t nesterov;
  float beta;
  float* partials;
  int32_t tile_start[kMaxBatch + 1];
  MomMat mat[kMaxBatch];
};

// ------------------------------------------------------- norm finalise (K2)
struct NormBatch {
  int32_t n;
  int32_t first;       // global index of mat 0 of this batch
  float eps;
  int32_t pad;
  const float* partials;
  float2* norm;        // {sum of squares, 1/(sqrt(sum)+eps)} per matrix
  int32_t start[kMaxBatch + 1];   // partial slots of matrix i: [start[i], start[i+1])
};

// ------------------------------------------------- Newton-Schulz GEMMs (K3-K5)
enum GemmMode : int32_t {
  kGram = 0,         // A = scale * X X^T               (X: K-major operand twice); also a plain
                     // product of two symmetric matrices (Gram-space program)
  kPoly = 1,         // B = b*A + c * A A               (A symmetric: K-major twice)
  kUpdate = 2,       // X' = scale * (a*X + B X)        (B K-major, X MN-major)
  kUpdateFinal = 3,  // same, written to the caller's update buffer
  kPolyI = 4,        // P = a*I + b*A + c * A A          (Gram-space program)
  kFinalQ = 5,       // X = scale * Q X0, written to the caller's update buffer (Gram-space program)
};

// The largest step count the Gram-space program runs (more steps take the
// standard program): its error stays at the standard program's for up to 5.
constexpr int kGramSpaceMaxSteps = 5;

// One matrix of a Newton-Schulz launch: its workspace buffers and the tiling
// of its three products.
struct NsMat {
  uint8_t* x[2];         // blocked bf16 iterates (s_pad x l_pad): iteration i reads x[i & 1], writes x[(i + 1) & 1]
  uint8_t* a;            // blocked bf16 A = X X^T (s_pad x s_pad)
  uint8_t* b;            // blocked bf16 B = b A + c A A
  void* out;             // the caller's update at the shard offset (may be null)
  void* w;               // apply: the weights at the shard offset, else null
  int32_t s_pad, l_pad;
  int32_t s, l;          // true short / long side
  int32_t tiles_sym;     // Gram / polynomial: pair tiles on or above the diagonal (256 or 128 wide)
  int32_t gram_space;    // 1: the Gram-space program (below), 0: the standard one
  uint8_t* c;            // Gram-space: blocked bf16 C = P A (s_pad x s_pad)
  uint8_t* q[2];         // Gram-space: blocked bf16 Q ping-pong (Q_0 = P_0 is written to q[0])
  int32_t tiles_m, tiles_n;   // update: 256-row pair tiles, 256 (or 128, narrow) columns wide
  int32_t n_last;        // update: width of the last column tile
  int32_t norm_idx;      // index into the norm table
  int32_t transposed;    // final update: stored matrix is l x s
  int32_t vec_ok;        // final update: stored rows start 16-byte aligned (offset and row length multiples of 8)
  float lr_scale;        // apply: lr * shape scale of this matrix
};

// One launch runs the products [phase_begin, phase_end) of the sequence
//   for it in 0 .. ns_steps-1: products 3 it, 3 it + 1, 3 it + 2
//   then product 3 ns_steps (Gram-space matrices only)
// over up to kMaxBatch matrices.  A matrix runs one of two programs that give
// the same update in exact arithmetic:
//   standard:     A = X X^T;  B = b A + c A A;  X <- a X + B X           (per iteration)
//   Gram-space:   iteration 0: A_0 = X0 X0^T, P_0 = a I + b A_0 + c A_0 A_0, C_0 = P_0 A_0;
//                 iteration k: A_k = C_{k-1} P_{k-1}, P_k = a I + b A_k + c A_k A_k,
//                              C_k = P_k A_k (not in the last), Q_k = P_k Q_{k-1} (Q_0 = P_0);
//                 then X = Q_{T-1} X0
// (X_{k+1} = P_k X_k, so A_{k+1} = P_k A_k P_k and X_T = P_{T-1} .. P_0 X0).
// Its tiles form one list, product-major (tile_begin .. tile_end-1 of the
// whole sequence's list), handed out in list order to whichever CTA pair asks
// next: iteration blocks of iter_tiles tiles, then the final Gram-space
// products from final_start.  Inside product k of an iteration (k = 3: the
// final block), matrix order[k][j] holds tiles [tile_start[k][j],
// tile_start[k][j+1]) after mode_start[k].  A Gram-space matrix's product 2
// holds its C tiles then its Q tiles; those that do not exist (Q in
// iteration 0, C in the last) are null tiles, taken and skipped.  A tile may
// start once every tile of the earlier products of its matrix in this launch
// has been stored: done[matrix] counts the epilogue warps that finished one.
struct NsBatch {
  int32_t n;
  int32_t ns_steps;
  int32_t phase_begin, phase_end;
  int32_t tile_begin, tile_end;
  int32_t stall_tile;    // test hook: this tile's dependency target is never reached (-1: none)
  int32_t iter_tiles;    // tiles of one iteration (three products, all matrices)
  int32_t final_start;   // first tile of the final Gram-space products (ns_steps * iter_tiles)
  int32_t mode_start[3];
  int32_t narrow;        // a launch with few tiles per iteration (its pairs take one tile at a time)
  int32_t narrow_mask;   // bit k: product k (kGram, kPoly, kUpdate) uses tiles 256 x 128 instead of 256 x 256
  int32_t out_bf16;      // final update dtype
  int32_t w_bf16;        // apply: weight dtype
  float a, b, c;
  float decay;           // apply: 1 - lr * weight_decay
  const float2* norm;
  const uint8_t* ws;     // workspace base: tensor-copy row y is byte 128 y of it
  int32_t* status;       // device status word (first wait that gave up)
  uint64_t wait_limit_ns;  // every wait of the launch gives up after this long (ns_wait_limit_ns)
  int32_t* next_tile;    // tiles handed out so far (dynamic schedule), zeroed before the launch
  int32_t* done;         // per matrix of the launch, zeroed before it
  int32_t tile_start[4][kMaxBatch + 1];
  uint8_t order[4][kMaxBatch];
  NsMat mat[kMaxBatch];
};
static_assert(kMaxBatch <= 256, "matrix order is stored in bytes");
static_assert(sizeof(NsBatch) < 32000, "kernel parameter limit");

// ------------------------------------------------------------ emit (T = 0)
struct EmitMat {
  const uint8_t* y;
  void* out;
  int64_t rows, cols;
  int32_t s_pad, tiles_j;
  int32_t transposed, norm_idx;
};
struct EmitBatch {
  int32_t n;
  int32_t out_bf16;
  const float2* norm;
  int32_t tile_start[kMaxBatch + 1];
  EmitMat mat[kMaxBatch];
};

// ------------------------------------------- owner segments (reduce / gather)
constexpr int kMaxSegBatch = 256;  // segments per launch
constexpr int kMaxSources = 64;    // source buffers (simulated ranks)
constexpr int kSegChunk = 2048;    // elements per CTA (256 threads x 8)
struct SegDesc {
  int64_t src_offset, dst_offset, numel;
  int32_t src_index;
  int32_t pad;
};
struct SegBatch {
  int32_t n;
  int32_t mode;          // 0: reduce over all sources in order; 1: gather from src[src_index]
  int32_t n_src;
  int32_t src_bf16;
  int32_t dst_bf16;
  int32_t pad;
  void* dst;
  const void* src[kMaxSources];
  int32_t chunk_start[kMaxSegBatch + 1];
  SegDesc seg[kMaxSegBatch];
};

// Status word written by a kernel that gives up on a bounded wait: the first
// one records (product index << 8) | role, role one of these.
enum WaitRole : int32_t {
  kRoleStageFree = 1,   // producer: a pipeline stage to refill
  kRoleStageFull = 2,   // MMA issuer: a stage's operands
  kRoleAccFree = 3,     // MMA issuer: an accumulator the epilogue has drained
  kRoleAccFull = 4,     // epilogue: a finished accumulator
  kRoleDependency = 5,  // producer or scheduler, or a role waiting behind the producer: earlier products of the tile's matrix
  kRoleTileFree = 7,    // scheduler: a ring slot every reader has taken
  kRoleTileFull = 8,    // producer, MMA issuer, epilogue: the next tile index
};

cudaError_t launch_momentum(const MomBatch& b, int total_tiles, cudaStream_t s);

// Every host-side check of an owner step's arguments except those of the
// workspace, without touching a device; *workspace_bytes (may be null)
// receives the scratch the step needs (0 for an empty owner set or an error).
int check_step_args(const mfsdp_matrix_shard* shards, int32_t n_shards, const void* grad, int32_t grad_dtype,
                    const float* momentum, const void* update, int32_t update_dtype, int64_t numel, double beta,
                    int32_t nesterov, int32_t ns_steps, double a, double b, double c, double eps,
                    size_t* workspace_bytes);
cudaError_t launch_norm_finalize(const NormBatch& b, cudaStream_t s);
cudaError_t launch_emit(const EmitBatch& b, int total_tiles, cudaStream_t s);
cudaError_t launch_ns(const NsBatch& b, size_t ws_bytes, cudaStream_t s);
cudaError_t launch_segments(const SegBatch& b, int total_chunks, cudaStream_t s);
// fp32 scalars of one AdamW step, formed in double on the host.
struct AdamScalars {
  float decay;         // 1 - lr*wd
  float beta1, beta2;
  float omb1, omb2;    // 1 - beta1, 1 - beta2
  float step_size;     // lr / (1 - beta1^step)
  float inv_sqrt_bc2;  // 1 / sqrt(1 - beta2^step)
  float eps;
};
cudaError_t launch_adamw(float* p, const float* g, float* m, float* v, int64_t n, const AdamScalars& k,
                         cudaStream_t s);

}  // namespace mfsdp
