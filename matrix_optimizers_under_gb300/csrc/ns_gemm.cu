// Newton-Schulz products on 5th-generation tensor cores (tcgen05 / TMEM): every
// product of every iteration, for every matrix of an owner set, in one launch.
//
// MatrixFSDP: Communication-Free Matrix Optimizers Under ZeRO-3 Parameter
// Sharding -- Abstract: Muon orthogonalises each owned matrix with
// Newton-Schulz locally on its owner.  Muon's quintic iteration on the short
// side (X is s x l):
//     A = X X^T              (kGram,   K = l)
//     B = b A + c A A        (kPoly,   K = s; A is symmetric so A A = A A^T)
//     X <- a X + B X         (kUpdate, K = s)
// with the Frobenius prescale 1/(||U||+eps) folded into the first iteration's
// epilogues (A scaled by its square, the new X by it).  A and B are symmetric:
// their products compute only the tiles on or above the diagonal of 256 x 256
// blocks (~53 % of the dense FLOPs), and the workspace keeps only those blocks.
// An operand block below that diagonal is read from the stored block across
// it, as the MN-major image of its transpose (the tensor copies and the MMA
// read either form; a diagonal 256 x 256 block is computed and stored whole,
// so it needs none): every product reads exactly the values it would read
// from the full matrix, and no epilogue writes a transposed copy.  A pair's
// tile is 256 x 256, or 256 x 128 ("narrow") for a product with fewer
// full-width tiles than CTA pairs in a launch with few tiles per iteration,
// where the chain of dependent products sets the time; each output element
// sums the same products in the same order at either width.
//
// A matrix with l >= 2s runs the same iteration in Gram space instead: with
// P_k = a I + b A_k + c A_k A_k, X_{k+1} = P_k X_k, so it iterates the s x s
// matrices A_{k+1} = (P_k A_k) P_k and Q_k = P_k Q_{k-1} and multiplies X_0 by
// Q_{T-1} once at the end.  All of them are polynomials in A_0, so every one
// of these products is symmetric and stored like A; the long K = l appears
// only in A_0 = X_0 X_0^T and the final Q X_0.  Products that read a diagonal
// 256 x 256 block as their B operand read it as columns, so that a block that
// is symmetric only up to rounding still gives the true product.  A
// contraction over the short side stops at s rounded up to 128: beyond it the
// operands' padding is zero where it meets.
//
// Operands live in the workspace in a blocked layout whose every 1 KB atom
// (8 rows x 64 bf16 columns) is already in the UMMA 128-byte-swizzle order, with
// atoms of one 64-column block contiguous.  So a CTA's share of a pipeline
// stage is one 16 KB run of rows per column block for each operand (for an
// MN-major operand, one 16 KB run of 128 K rows per 64-column block),
// and a tensor copy through a map that views the whole
// workspace as 128-byte rows lands it in shared memory byte for byte, ready
// for tcgen05.mma.  Two maps of that one view (boxes of 128 and 64 rows: 16 KB
// runs, and the 8 KB B halves of 128-column tiles) serve any mix of shapes in
// one launch, and the same stored X serves as the K-major operand of the Gram
// product and the MN-major operand of the update.
//
// One launch runs every product of every iteration for up to kMaxBatch
// matrices.  Its tiles form one product-major list (all Gram tiles of
// iteration 0, then all polynomial tiles, ...).  Persistent CTA pairs (one CTA
// per SM) take tiles from it in list order through a global counter, so the
// tiles in flight are always a contiguous window of the list, which keeps the
// operands the pairs share in L2.  A tile may start only once the earlier
// products of its own matrix are stored: each epilogue warp that stores its
// share of a tile adds one to the matrix's completion counter (release).  In
// each pair a scheduler warp of the even CTA takes the next index and hands
// the tile to its own CTA's roles and to the odd CTA's scheduler (a remote
// store and mbarrier arrive), which passes it to the odd CTA's roles; each CTA
// passes tiles through a small ring in shared memory.  The scheduler reads
// the counter of the tile's matrix once (acquire): a tile whose earlier
// products are all stored goes out "ready", any other marked "wait", and then
// both producers of the pair poll the counter (acquire) until it covers every
// tile of the earlier products before their tensor copies -- a hand-over
// across the pair costs a cluster-scope release (~850 cycles on GB300), which
// would otherwise lie between a product's last store and the next product's
// first copies.  Each producer tells its CTA's other roles through an
// mbarrier.  The scheduler takes the next index only once the tile may start
// (it polls the counter too, or in a small launch waits for its producer), so
// a pair that cannot start a tile takes no more of the list; otherwise it
// runs ahead of the roles, so taking a tile costs the pipeline nothing while
// work is ready.  Small matrices run ahead
// through their iterations while large ones fill the machine, with no launch
// gap or tail between products.  Every dependency points to an earlier
// position of the list and tiles are taken in list order, so the lowest
// unfinished tile belongs to a running pair and can always proceed.
//
// A pair computes a 256 x N tile with the pair MMA (tcgen05 cta_group::2,
// M = 256): each CTA holds 128 rows of A and half of B's N columns in its own
// shared memory, and its 128 output rows in its own TMEM.  In each CTA, warp 0
// (one lane) streams K in 128-element stages (two column blocks of the layout)
// through a 3-deep mbarrier ring of 64 KB stages; its tensor copies complete on
// the even CTA's full barrier
// (cta_group::2 copies), which the even producer arms with both CTAs' bytes.
// The even CTA's warp 1 (one lane) issues 256 x N x 16 pair UMMAs into one of
// two 256-column accumulators and frees each stage in both CTAs with one
// multicast commit.  Warps 2-9 of both CTAs drain the other accumulator: two
// halves of four warps (one per TMEM lane quadrant), each half owning half the
// tile's columns.  A half moves each 128-row x 64-column block of its input
// (A or X) and output through a 16 KB stage in shared memory with 16-byte
// accesses at consecutive addresses (the block is one contiguous 16 KB run in
// the workspace), while each thread reads its accumulator row (tcgen05.ld),
// its input row from the stage, applies the fused epilogue in fp32 and writes
// bf16 back into the stage -- or, on the last iteration, the update in the
// caller's dtype and layout, transposed back for tall matrices -- and the
// accumulator goes back to the even CTA's issuer after its last read.  So one
// tile's epilogue runs under the next tile's main loop.  Every wait is
// bounded: on expiry the CTA records which wait gave up in the status word,
// every other CTA sees the word and stops too, and each drains what it issued,
// frees TMEM and returns.
//
// Bounds of every tensor copy (the long side is padded to a multiple of 128
// and the short side to a multiple of 256; K, l_pad or s rounded up to 128,
// is a multiple of 128 and at most the operand's padded width, and a stage
// covers column blocks 2kb and 2kb+1): a CTA's A rows in column block c
// start at c*s_pad*128 + (mc/8)*1024 and span 16 KB, ending at most at
// (K/64-1)*s_pad*128 + (s_pad-128)*128 + 16384 = K*s_pad*2, the end of the
// operand; its K-major B half likewise ends at most at (K/64-1)*s_pad*128 +
// n0*128 + N*128 <= K*s_pad*2 since n0 + N <= s_pad; the MN-major X runs
// (column block n0/64 + j, K rows 128kb..128kb+127, 16 KB) end at most at
// (l_pad/64-1)*s_pad*128 + (s_pad/128-1)*16384 + 16384 = l_pad*s_pad*2, the
// end of X.  Every run starts on a 128-byte row of the map, so its x
// coordinate is 0.
#include <cuda.h>
#include <cuda_bf16.h>

#include <climits>
#include <mutex>

#include "mfsdp_internal.h"
#include "ptx.cuh"

namespace mfsdp {
namespace {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: the floor of every wait's limit, and the drains' limit
constexpr uint32_t kAccCols = 256;     // one fp32 accumulator of 128 lanes x 256 columns
constexpr uint32_t kTmemCols = 512;    // two accumulators: epilogue of tile i overlaps the MMAs of tile i+1
constexpr int32_t kArrivalsPerTile = 2 * kEpilogueWarps;   // completion-counter adds per pair tile
constexpr int kTileRing = 4;           // ready tiles handed from a CTA's scheduler to its roles
constexpr uint32_t kTileReaders = 2 + kEpilogueWarps;   // producer, MMA issuer, epilogue warps
constexpr int kPairRing = 4;           // tiles handed from the even CTA's scheduler to the odd one's
// Set in a handed-out tile index when the scheduler found the tile's earlier
// products not yet stored: the producers then wait for them themselves.
constexpr int32_t kPollBit = 1 << 30;

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

// The epilogue stages each 128-row x 64-column block of a CTA's tile in
// shared memory, in the layout the block has in the workspace: there it is one
// contiguous 16 KB run (16 atoms of one column block).  Its input (A or X) is
// read from global memory, and its output written back, by the 128 threads of
// a half of the epilogue warps with 16-byte accesses at consecutive addresses
// (each warp access covers 512 contiguous bytes); a thread of the tile's row
// reads and writes its own 16-byte chunks in shared memory, where the atom
// swizzle spreads a warp's 32 rows over all banks.  (Each thread reading and
// writing its own row straight from global memory touched 32 lines per warp
// access, half of each sector, and cost ~6 us per tile in a latency-bound
// owner set.)
constexpr int kRunChunks = kStageOutBytes / 16 / 128;   // 16-byte chunks per thread of a 16 KB run (8)

// The input run, read from L2 (ld.global.cg: it was written by other CTAs
// earlier in this launch, so never from a possibly stale L1 line).
__device__ __forceinline__ void load_run(const uint8_t* run, int k, uint4 (&w)[kRunChunks]) {
#pragma unroll
  for (int i = 0; i < kRunChunks; ++i) w[i] = __ldcg(reinterpret_cast<const uint4*>(run) + k + 128 * i);
}
__device__ __forceinline__ void put_run(uint8_t* stage, int k, const uint4 (&w)[kRunChunks]) {
#pragma unroll
  for (int i = 0; i < kRunChunks; ++i) reinterpret_cast<uint4*>(stage)[k + 128 * i] = w[i];
}
__device__ __forceinline__ void store_run(uint8_t* run, const uint8_t* stage, int k) {
#pragma unroll
  for (int i = 0; i < kRunChunks; ++i)
    reinterpret_cast<uint4*>(run)[k + 128 * i] = reinterpret_cast<const uint4*>(stage)[k + 128 * i];
}

// Byte offset in a staged block of the q-th 16-byte chunk of columns
// [c, c + 32) (c = 0 or 32 within the block) of block row r (0..127).
__device__ __forceinline__ uint32_t stage_off(int r, int c, int q) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((((c >> 3) + q) ^ (r & 7)) << 4));
}

// Unpack 32 bf16 (four 16-byte chunks) into fp32.
__device__ __forceinline__ void unpack_bf16x32(const uint4 (&w)[4], float (&x)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    x[8 * q + 0] = bf_lo(w[q].x); x[8 * q + 1] = bf_hi(w[q].x);
    x[8 * q + 2] = bf_lo(w[q].y); x[8 * q + 3] = bf_hi(w[q].y);
    x[8 * q + 4] = bf_lo(w[q].z); x[8 * q + 5] = bf_hi(w[q].z);
    x[8 * q + 6] = bf_lo(w[q].w); x[8 * q + 7] = bf_hi(w[q].w);
  }
}

__device__ __forceinline__ void stage_chunk(uint8_t* stage, int r, int c, const float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 w;
    w.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
    w.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
    w.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
    w.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
    *reinterpret_cast<uint4*>(stage + stage_off(r, c, q)) = w;
  }
}

// One element of the final step at a stored position: the update O (when the
// caller asked for it) and, when applying, W <- decay * W - lr_scale * O.
__device__ __forceinline__ void final_elem(const NsMat& d, const NsBatch& p, int64_t o, float v) {
  if (d.out) {
    if (p.out_bf16) static_cast<__nv_bfloat16*>(d.out)[o] = __float2bfloat16_rn(v);
    else static_cast<float*>(d.out)[o] = v;
  }
  if (d.w) {
    if (p.w_bf16) {
      __nv_bfloat16* w = static_cast<__nv_bfloat16*>(d.w) + o;
      *w = __float2bfloat16_rn(fmaf(-d.lr_scale, v, p.decay * __bfloat162float(*w)));
    } else {
      float* w = static_cast<float*>(d.w) + o;
      *w = fmaf(-d.lr_scale, v, p.decay * *w);
    }
  }
}

// The final update of a tall matrix (stored l x s, X = its transpose) writes
// through the epilogue half's stage: each of the half's 128
// threads holds X row m = mc + r for 32 consecutive X columns [n, n + 32),
// i.e. one element of 32 consecutive stored rows, so the chunk is put into
// the stage transposed (stored row j, then the 128 stored columns mc ..
// mc + 127), and after the half's meeting copied out with 16-byte stores
// along the stored rows -- instead of a 2-byte store per element, 64 bytes
// per warp access.  Needs the stored rows to start 16-byte aligned
// (vec_ok: offset and s multiples of 8); the stage's bytes per element are
// those of the output (a 32 x 128 chunk: 8 KB bf16, 16 KB fp32).
__device__ __forceinline__ void stage_final_t(uint8_t* stage, int r, const float (&v)[32], bool bf16) {
  if (bf16) {
    __nv_bfloat16* st = reinterpret_cast<__nv_bfloat16*>(stage);
#pragma unroll
    for (int j = 0; j < 32; ++j) st[j * 128 + r] = __float2bfloat16_rn(v[j]);
  } else {
    float* st = reinterpret_cast<float*>(stage);
#pragma unroll
    for (int j = 0; j < 32; ++j) st[j * 128 + r] = v[j];
  }
}
// ... copied out by thread k of the half: stored rows n .. n + 31 (those below
// l), columns mc .. mc + 127 (the 16-byte pieces below s).
__device__ __forceinline__ void store_final_t(const NsMat& d, const NsBatch& p, const uint8_t* stage, int mc, int n,
                                              int k) {
  const int es = p.out_bf16 ? 2 : 4;
  const int row_pieces = 128 * es / 16;                      // 16-byte pieces of one stored row's 128 columns
  const int pieces = 32 * row_pieces;
  for (int c = k; c < pieces; c += 128) {
    const int j = c / row_pieces, col = (c - j * row_pieces) * (16 / es);
    if (n + j >= d.l || mc + col >= d.s) continue;
    const int64_t o = (int64_t)(n + j) * d.s + mc + col;
    *reinterpret_cast<uint4*>(static_cast<uint8_t*>(d.out) + o * es) =
        *reinterpret_cast<const uint4*>(stage + (size_t)c * 16);
  }
}

// Final update for 32 consecutive X columns [n, n+32) of X row m, in the
// caller's layout: stored (m, n) when not transposed, (n, m) otherwise.
__device__ __forceinline__ void store_final(const NsMat& d, const NsBatch& p, int m, int n, const float (&v)[32]) {
  if (m >= d.s) return;
  if (!d.transposed) {
    const int64_t row0 = (int64_t)m * d.l;
    if (d.vec_ok && !d.w && n + 32 <= d.l) {
      if (p.out_bf16) {
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
      for (int j = 0; j < 32; ++j)
        if (n + j < d.l) final_elem(d, p, row0 + n + j, v[j]);
    }
  } else {
    // stored matrix is l x s: element (n + j, m); the warp's 32 rows m are
    // contiguous in memory, so each j is one coalesced store.
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (n + j < d.l) final_elem(d, p, (int64_t)(n + j) * d.s + m, v[j]);
  }
}

struct Tile {
  int mi;        // matrix index in the batch
  int phase;     // product index in the sequence: 3 * iteration + product (3 * ns_steps: final Gram-space)
  int mode;      // a GemmMode
  bool first;    // first iteration: fold the Frobenius prescale into the epilogue
  bool symmetric;
  bool a_sym;    // A operand is a symmetric product stored as its upper 256 x 256 blocks
  bool b_sym;    // the K-major B operand likewise
  bool b_mn;     // B operand is the MN-major X (update-like products)
  bool zero;     // the matrix's momentum is exactly zero: no products
  bool null;     // a Gram-space product that does not exist (Q in iteration 0, C in the last): skipped
  bool last;     // the matrix's last product: nothing waits for it
  int m0, n0;    // origin of the pair's 256-row output tile
  int mc;        // this CTA's 128 rows: [mc, mc + 128)
  int N;         // tile width (256, or 128 for the last column tile)
  int k_blocks;  // K / kBlockK
  int s_pad;     // the matrix's padded short side: rows of every operand's column block
  int32_t need;  // completions of this matrix's earlier products (this launch) to wait for
  const uint8_t* a_op;   // blocked bf16 source of UMMA operand A (rows m)
  const uint8_t* b_op;   // blocked bf16 source of UMMA operand B
  const uint8_t* c_in;   // blocked bf16 epilogue input (A for kPoly / kPolyI, X for the update)
  void* out;             // blocked bf16 output, or the caller's buffer (final update)
};
static_assert(sizeof(Tile) % 8 == 0 && alignof(Tile) == 8, "tiles cross the pair as 8-byte words");

// Tiles of a matrix's products [0, ph) that publish a completion: whole
// iterations, then the products of the current one before it, less (Gram-space)
// the null tiles among them.
__device__ __forceinline__ int tiles_before(const NsBatch& p, const NsMat& d, int ph) {
  if (!d.gram_space) {
    const int per_iter = 2 * d.tiles_sym + d.tiles_m * d.tiles_n;
    return (ph / 3) * per_iter + (ph % 3) * d.tiles_sym;
  }
  const int sym = d.tiles_sym;
  int n = (ph / 3) * 4 * sym + (ph % 3 >= 1 ? sym : 0) + (ph % 3 >= 2 ? sym : 0);
  if (ph > 2) n -= sym;                        // Q of iteration 0
  if (ph > 3 * p.ns_steps - 1) n -= sym;       // C of the last iteration
  return n;
}

// Tile t of the sequence's list.  Symmetric products: 256 x 256 tiles on or
// above the diagonal, row pair-block I holding tiles I .. nb2-1; update-like
// products: 256-row tiles, rows fastest (neighbours share B-operand columns).
__device__ __forceinline__ Tile decode_tile(const NsBatch& p, int t, uint32_t rank) {
  Tile r;
  int it, prod, rem;
  if (t < p.final_start) {
    it = t / p.iter_tiles;
    rem = t - it * p.iter_tiles;
    prod = rem >= p.mode_start[2] ? 2 : (rem >= p.mode_start[1] ? 1 : 0);
    rem -= p.mode_start[prod];
  } else {
    it = p.ns_steps;
    prod = 3;
    rem = t - p.final_start;
  }
  const int k = find_mat(p.tile_start[prod], p.n, rem);
  r.mi = p.order[prod][k];
  int local = rem - p.tile_start[prod][k];
  const NsMat& d = p.mat[r.mi];
  const bool last_it = it == p.ns_steps - 1;
  r.phase = prod == 3 ? 3 * p.ns_steps : 3 * it + prod;
  r.first = false;
  r.null = false;
  r.symmetric = true;
  r.a_sym = r.b_sym = r.b_mn = false;
  r.c_in = nullptr;
  // K = s: the operands' rows and columns past s hold zeros where they meet
  // (the Gram-space P and Q carry a on their padded diagonal, which only ever
  // multiplies zero rows into padded rows), so the K loop ends at the last
  // 128-wide block that holds a real row.
  r.k_blocks = (d.s + kBlockK - 1) / kBlockK;
  if (!d.gram_space) {
    uint8_t* xc = d.x[it & 1];
    r.first = it == 0;
    r.last = prod == kUpdate && last_it;
    if (prod == kGram) {
      r.mode = kGram;
      r.a_op = xc; r.b_op = xc; r.out = d.a;
      r.k_blocks = d.l_pad / kBlockK;
    } else if (prod == kPoly) {
      r.mode = kPoly;
      r.a_op = d.a; r.b_op = d.a; r.c_in = d.a; r.out = d.b;
      r.a_sym = r.b_sym = true;
    } else {
      r.mode = last_it ? kUpdateFinal : kUpdate;
      r.a_op = d.b; r.b_op = xc; r.c_in = xc;
      r.out = last_it ? d.out : static_cast<void*>(d.x[(it + 1) & 1]);
      r.symmetric = false;
      r.a_sym = r.b_mn = true;
    }
  } else {
    // Gram-space: P_0 is kept in q[0] (it is Q_0), P_k (k >= 1) in b.
    uint8_t* const p_it = it == 0 ? d.q[0] : d.b;
    r.last = prod == 3;
    if (prod == 0) {
      r.mode = kGram;
      if (it == 0) {                                   // A_0 = X0 X0^T (prescaled)
        r.first = true;
        r.a_op = d.x[0]; r.b_op = d.x[0];
        r.k_blocks = d.l_pad / kBlockK;
      } else {                                         // A_it = C_{it-1} P_{it-1}
        r.a_op = d.c; r.b_op = it == 1 ? d.q[0] : d.b;
        r.a_sym = r.b_sym = true;
      }
      r.out = d.a;
    } else if (prod == 1) {                            // P_it = a I + b A + c A A
      r.mode = kPolyI;
      r.a_op = d.a; r.b_op = d.a; r.c_in = d.a; r.out = p_it;
      r.a_sym = r.b_sym = true;
    } else if (prod == 2) {
      r.mode = kGram;
      r.a_sym = r.b_sym = true;
      if (local < d.tiles_sym) {                       // C_it = P_it A_it
        r.a_op = p_it; r.b_op = d.a; r.out = d.c;
        r.null = last_it;
      } else {                                         // Q_it = P_it Q_{it-1}
        local -= d.tiles_sym;
        r.a_op = p_it; r.b_op = d.q[(it - 1) & 1]; r.out = d.q[it & 1];
        r.null = it == 0;
      }
    } else {                                           // X = Q_{T-1} X0, prescaled
      r.mode = kFinalQ;
      r.a_op = d.q[(p.ns_steps - 1) & 1]; r.b_op = d.x[0]; r.out = d.out;
      r.symmetric = false;
      r.a_sym = r.b_mn = true;
    }
  }
  // tile columns: 128 in a narrow launch for a product class with few tiles
  const int width = (p.narrow_mask >> (r.symmetric ? kGram : kUpdate)) & 1 ? kBlockN / 2 : kBlockN;
  if (r.symmetric) {
    // Row pair-block I holds the tiles of columns 256 I .. s_pad - 1: nb2 - I
    // of them, or twice that for narrow tiles.
    const int nb2 = d.s_pad / kPairM, per = kBlockN / width;
    int rem2 = local, I = 0;
    while (I < nb2 - 1 && rem2 >= per * (nb2 - I)) {
      rem2 -= per * (nb2 - I);
      ++I;
    }
    r.m0 = I * kPairM;
    r.n0 = I * kPairM + rem2 * width;
    r.N = width;
  } else {
    const int mt = local % d.tiles_m, nt = local / d.tiles_m;
    r.m0 = mt * kPairM;
    r.n0 = nt * width;
    r.N = (nt == d.tiles_n - 1) ? d.n_last : width;
  }
  r.mc = r.m0 + (int)rank * kBlockM;
  r.s_pad = d.s_pad;
  r.zero = p.norm[d.norm_idx].x == 0.0f;
  r.need = kArrivalsPerTile * (tiles_before(p, d, r.phase) - tiles_before(p, d, p.phase_begin));
  return r;
}

// Operand sources of stage kb of a tile (bounds: see the file header).
__device__ __forceinline__ const uint8_t* a_block(const Tile& tl, int kb, size_t kstride) {
  return tl.a_op + (size_t)kb * kstride + (size_t)(tl.mc >> 3) * 1024;
}
// K-major B: rows [n0 + half * N/2, + N/2).
__device__ __forceinline__ const uint8_t* b_half_kmajor(const Tile& tl, int kb, size_t kstride, uint32_t half) {
  return tl.b_op + (size_t)kb * kstride + (size_t)((tl.n0 + (int)half * (tl.N >> 1)) >> 3) * 1024;
}
// MN-major X: 64-column block n0/64 + j, K rows [64 kb, 64 kb + 64).
__device__ __forceinline__ const uint8_t* b_block_mn(const Tile& tl, int kb, size_t kstride, int j) {
  return tl.b_op + (size_t)((tl.n0 >> 6) + j) * kstride + (size_t)kb * 8 * 1024;
}
// The symmetric products are stored as their 128 x 128 blocks (r, c) with
// c/2 >= r/2 only (on or above the diagonal of 256 x 256 blocks); a block
// below it stands for the transpose of its mirror image, while a diagonal
// 256 x 256 block is stored whole, as computed.  A product of two such
// matrices Y Z takes row m of Y and column n of Z for each stage kb (K columns
// [128 kb, 128 kb + 128)):
//   A operand (rows of Y): the stored rows where K's 256-block is on or right
//     of the rows' one, else the MN-major image of the stored block across
//     the diagonal;
//   B operand (columns of Z, as rows of its transpose): the MN-major image of
//     the stored block where K's 256-block is on or above the columns' one,
//     else the stored rows of the block across the diagonal.
// (For an exactly symmetric Z -- the standard form's A -- both images of the
// diagonal block hold the same values.  The Gram-space form's products P A,
// C P and P Q are symmetric only up to rounding, and reading the diagonal
// blocks as columns makes each one the true product of the stored matrices,
// as its polynomial needs.)  Both CTAs of the pair decide alike, since their
// rows, and their halves of the tile's columns, share one 256-block.
__device__ __forceinline__ bool a_trans(const Tile& tl, int kb) { return tl.a_sym && (kb >> 1) < (tl.m0 >> 8); }
__device__ __forceinline__ bool b_trans(const Tile& tl, int kb) { return tl.b_sym && (kb >> 1) <= (tl.n0 >> 8); }
// Transposed A: 64-column block mc/64 + j of the stored matrix, rows
// [128 kb, 128 kb + 128): one 16 KB run.
__device__ __forceinline__ const uint8_t* a_block_t(const Tile& tl, int kb, size_t kstride, int j) {
  return tl.a_op + (size_t)((tl.mc >> 6) + j) * kstride + (size_t)kb * 16384;
}

// Row of the workspace tensor map (128-byte rows) where a blocked run starts.
__device__ __forceinline__ int32_t ws_row(const NsBatch& p, const uint8_t* src) { return (int32_t)((src - p.ws) >> 7); }

__device__ __forceinline__ int32_t wait_code(int phase, int role) { return (phase << 8) | role; }

// What a bounded wait needs: the CTA's abort flag (another role of this CTA
// gave up), the launch's status word (another CTA recorded a failure) and the
// launch's wait limit (NsBatch::wait_limit_ns).
struct Abort {
  volatile int* flag;
  int32_t* status;
  uint64_t limit_ns;
};

// Called between polls of a wait: true when the wait must be abandoned --
// another role of this CTA gave up, another CTA recorded a failure, or this
// wait has run for the launch's limit (then it records `code`).
__device__ __forceinline__ bool give_up(const Abort& ab, uint64_t t0, int32_t code) {
  if (*ab.flag) return true;
  if (*reinterpret_cast<volatile int32_t*>(ab.status) != 0) {
    *ab.flag = 1;
    return true;
  }
  if (ptx::globaltimer_ns() - t0 > ab.limit_ns) {
    *ab.flag = 1;
    atomicCAS(ab.status, 0, code);
    return true;
  }
  return false;
}

// Bounded mbarrier wait.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, const Abort& ab, int32_t code) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (ptx::mbar_try_wait(bar, parity)) return true;
    if (give_up(ab, t0, code)) return false;
  }
}

// Bounded wait until a matrix's completion counter reaches `need` (acquire:
// the stores it counts are visible to this thread afterwards).
__device__ __forceinline__ bool wait_done(const int32_t* ctr, int32_t need, const Abort& ab, int32_t code) {
  if (ptx::ld_acquire_gpu(ctr) >= need) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 8; ++i) {
      __nanosleep(64);
      if (ptx::ld_acquire_gpu(ctr) >= need) return true;
    }
    if (give_up(ab, t0, code)) return false;
  }
}

// Bounded wait on an mbarrier that another CTA of the pair arrives on
// (acquire at cluster scope).
__device__ __forceinline__ bool wait_cluster_or_abort(uint32_t bar, uint32_t parity, const Abort& ab, int32_t code) {
  if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
    if (give_up(ab, t0, code)) return false;
  }
}

// The four warps of one epilogue half meet on their mbarrier (every thread
// arrives, so each thread's shared-memory writes before it are visible to all
// of them after it).  Bounded like every other wait; false, warp-uniform, when
// the kernel is giving up.
__device__ __forceinline__ bool half_sync(uint32_t bar, uint32_t& phase, const Abort& ab, int32_t code) {
  ptx::mbar_arrive(bar);
  const bool ok = wait_or_abort(bar, phase & 1, ab, code);
  ++phase;
  return __all_sync(0xffffffffu, ok);
}

// A ring of tile indices: slot k holds the tiles of sequence numbers
// k, k + size, ...; full[k] (count 1) completes when the writer has stored
// it, empty[k] when every reader has taken it.  Each CTA's scheduler feeds
// its own roles through a CTA-local ring; the even CTA's scheduler feeds the
// odd one's through a ring in the odd CTA (remote store and arrive), whose
// empty barriers live in the even CTA.
struct Ring {
  uint32_t slot0;    // slot 0 (shared address, in the readers' CTA)
  uint32_t full0;    // full[0], in the readers' CTA
  uint32_t empty0;   // empty[0], in the writer's CTA
};

// CTA-local ring: the scheduler stores tile t into slot seq for this CTA's
// roles, with the tile decoded for this CTA (`tiles`, the ring's slots of
// decoded tiles; unused for the end marker).  Decoding reads the launch's
// tables from the kernel parameters at scattered offsets (~1800 cycles); the
// scheduler, which runs ahead of the roles, does it once per CTA, and the
// roles copy the result from shared memory.
__device__ __forceinline__ bool local_publish(const Ring& r, uint32_t seq, int32_t t, const Abort& ab,
                                              Tile* tiles, const Tile* tl) {
  const uint32_t k = seq % kTileRing, use = seq / kTileRing;
  if (!wait_or_abort(r.empty0 + 8u * k, (use & 1) ^ 1, ab, wait_code(0, kRoleTileFree))) return false;
  if (tl) tiles[k] = *tl;
  asm volatile("st.shared.s32 [%0], %1;" ::"r"(r.slot0 + 4u * k), "r"(t) : "memory");
  ptx::mbar_arrive(r.full0 + 8u * k);   // releases the stores (CTA scope)
  return true;
}

// A role reads the tile of sequence number seq from its CTA's ring (`poll`:
// whether kPollBit was set) ...
__device__ __forceinline__ bool local_peek(const Ring& r, uint32_t seq, int32_t& t, const Abort& ab,
                                           bool* poll = nullptr) {
  const uint32_t k = seq % kTileRing, use = seq / kTileRing;
  if (!wait_or_abort(r.full0 + 8u * k, use & 1, ab, wait_code(0, kRoleTileFull))) return false;
  int32_t v;
  asm volatile("ld.shared.s32 %0, [%1];" : "=r"(v) : "r"(r.slot0 + 4u * k) : "memory");
  if (poll) *poll = (v & kPollBit) != 0;
  t = v & ~kPollBit;
  return true;
}
// ... and gives the slot back (every reader of the CTA does, once per tile).
__device__ __forceinline__ void local_release(const Ring& r, uint32_t seq) {
  ptx::mbar_arrive(r.empty0 + 8u * (seq % kTileRing));
}
__device__ __forceinline__ bool local_take(const Ring& r, uint32_t seq, int32_t& t, const Abort& ab,
                                           bool* poll = nullptr) {
  if (!local_peek(r, seq, t, ab, poll)) return false;
  local_release(r, seq);
  return true;
}
// The decoded tile of sequence number seq (read between peek and release).
__device__ __forceinline__ Tile ring_tile(const Tile* tiles, uint32_t seq) { return tiles[seq % kTileRing]; }

// Pair ring, even CTA's scheduler side: stores tile t into the odd CTA's slot
// seq, with the tile decoded for the odd CTA (tl; null for the end marker)
// into the odd CTA's copy of `tiles` (shared address of slot 0 in this CTA).
__device__ __forceinline__ bool pair_publish(const Ring& r, uint32_t seq, int32_t t, const Abort& ab,
                                             uint32_t tiles, const Tile* tl) {
  const uint32_t k = seq % kPairRing, use = seq / kPairRing;
  if (!wait_cluster_or_abort(r.empty0 + 8u * k, (use & 1) ^ 1, ab, wait_code(0, kRoleTileFree)))
    return false;
  if (tl) {
    const uint32_t dst = ptx::mapa_shared(tiles + (uint32_t)sizeof(Tile) * k, 1);
    const uint64_t* w = reinterpret_cast<const uint64_t*>(tl);
#pragma unroll
    for (int i = 0; i < (int)(sizeof(Tile) / 8); ++i) ptx::st_shared_cluster_u64(dst + 8u * i, w[i]);
  }
  ptx::st_shared_cluster_s32(ptx::mapa_shared(r.slot0 + 4u * k, 1), t);
  ptx::mbar_arrive_cluster(ptx::mapa_shared(r.full0 + 8u * k, 1));   // releases the stores (cluster scope)
  return true;
}

// Pair ring, odd CTA's scheduler side: takes the tile of sequence number seq
// (its decoded form is then in slot seq % kPairRing of the pair's tiles).
__device__ __forceinline__ bool pair_take(const Ring& r, uint32_t seq, int32_t& t, const Abort& ab) {
  const uint32_t k = seq % kPairRing, use = seq / kPairRing;
  if (!wait_cluster_or_abort(r.full0 + 8u * k, use & 1, ab, wait_code(0, kRoleTileFull))) return false;
  asm volatile("ld.shared.s32 %0, [%1];" : "=r"(t) : "r"(r.slot0 + 4u * k) : "memory");
  return true;
}
// ... and frees its slot for the even CTA's scheduler (called after the tile
// has been passed on: the cluster-scope release stalls this thread).
__device__ __forceinline__ void pair_free(const Ring& r, uint32_t seq) {
  ptx::mbar_arrive_cluster(ptx::mapa_shared(r.empty0 + 8u * (seq % kPairRing), 0));
}

__global__ void __launch_bounds__(kGemmThreads, 1) ns_kernel(const __grid_constant__ NsBatch p,
                                                             const __grid_constant__ CUtensorMap tmap_8k,
                                                             const __grid_constant__ CUtensorMap tmap_16k) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ __align__(8) uint64_t tfull_bar[2];    // accumulator ready for the epilogue
  __shared__ __align__(8) uint64_t tempty_bar[2];   // accumulator drained, MMA may reuse it
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ __align__(8) uint64_t half_bar[2];     // the two halves of the epilogue warps meet
  __shared__ __align__(8) uint64_t ring_full[kTileRing];
  __shared__ __align__(8) uint64_t ring_empty[kTileRing];
  __shared__ int32_t ring_slot[kTileRing];
  __shared__ Tile ring_tiles[kTileRing];                    // the ring's tiles, decoded for this CTA
  __shared__ __align__(8) uint64_t dep_bar[kTileRing];     // tile seq's earlier products are stored (producer)
  __shared__ __align__(8) uint64_t pair_full[kPairRing];    // used in the odd CTA
  __shared__ __align__(8) uint64_t pair_empty[kPairRing];   // used in the even CTA
  __shared__ int32_t pair_slot[kPairRing];                  // used in the odd CTA
  __shared__ Tile pair_tiles[kPairRing];                    // used in the odd CTA: its decoded tiles
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();          // 0 or 1 within the CTA pair
  const uint32_t smem_base = (ptx::smem_u32(smem_raw) + 1023u) & ~1023u;
  constexpr uint16_t kPair = 0x3;                        // both CTAs of the cluster
  const Ring ring{ptx::smem_u32(&ring_slot[0]), ptx::smem_u32(&ring_full[0]), ptx::smem_u32(&ring_empty[0])};
  const Ring pair{ptx::smem_u32(&pair_slot[0]), ptx::smem_u32(&pair_full[0]), ptx::smem_u32(&pair_empty[0])};

  if (warp == 1) {
    // The pair's accumulators: one warp of each CTA allocates jointly.
    ptx::tmem_alloc_pair(ptx::smem_u32(&tmem_slot), kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(ptx::smem_u32(&full_bar[s]), 1);    // used in the even CTA: both CTAs' copies
      ptx::mbar_init(ptx::smem_u32(&empty_bar[s]), 1);   // the pair MMA's commit
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(ptx::smem_u32(&tfull_bar[a]), 1);
      ptx::mbar_init(ptx::smem_u32(&tempty_bar[a]), 2 * kEpilogueWarps);   // even CTA: both CTAs' epilogues
    }
    ptx::mbar_init(ptx::smem_u32(&drain_bar), 1);
    for (int h = 0; h < 2; ++h) ptx::mbar_init(ptx::smem_u32(&half_bar[h]), 4 * 32);
    for (int k = 0; k < kTileRing; ++k) {
      ptx::mbar_init(ptx::smem_u32(&ring_full[k]), 1);
      ptx::mbar_init(ptx::smem_u32(&ring_empty[k]), kTileReaders);
      ptx::mbar_init(ptx::smem_u32(&dep_bar[k]), 1);
    }
    for (int k = 0; k < kPairRing; ++k) {
      ptx::mbar_init(ptx::smem_u32(&pair_full[k]), 1);
      ptx::mbar_init(ptx::smem_u32(&pair_empty[k]), 1);
    }
    abort_flag = 0;
    ptx::fence_barrier_init();
    ptx::fence_proxy_async_smem();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync();    // both CTAs' barriers exist before any multicast or remote arrive
  ptx::tc_fence_after();
  const uint32_t tmem_base = tmem_slot;
  const Abort ab{&abort_flag, p.status, p.wait_limit_ns};

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      // This CTA loads its own 128 rows of A and its half of B's columns into
      // its own shared memory, as tensor copies of the workspace.  Every copy
      // of both CTAs completes on the even CTA's full barrier, which the even
      // producer arms with both CTAs' bytes: the pair MMA reads both halves.
      ptx::prefetch_tensormap(&tmap_8k);
      ptx::prefetch_tensormap(&tmap_16k);
      const uint64_t pol = ptx::policy_evict_last();
      uint32_t it = 0, seq = 0;
      bool ok = true;
      while (ok) {
        int32_t t;
        bool poll = false;
        ok = local_peek(ring, seq, t, ab, &poll);
        if (!ok || t >= p.tile_end) break;
        const Tile tl = ring_tile(ring_tiles, seq);
        local_release(ring, seq);
        // A tile whose earlier products were not all stored when the
        // scheduler took it: both producers of the pair wait (acquire) until
        // they are, so neither CTA's copies wait for a hand-over after the
        // last of them lands.  (Otherwise the scheduler's acquire reaches this
        // thread through the rings.)  dep_bar passes the wait on to this CTA's
        // epilogue (which reads those products too), MMA issuer and scheduler.
        const int32_t need = t == p.stall_tile ? INT32_MAX : tl.need;   // the test hook: a count never reached
        if (poll && !wait_done(p.done + tl.mi, need, ab, wait_code(tl.phase, kRoleDependency))) {
          ok = false;
          break;
        }
        ptx::mbar_arrive(ptx::smem_u32(&dep_bar[seq % kTileRing]));   // releases the acquire (CTA scope)
        ++seq;
        if (tl.zero || tl.null) continue;
        // The operands were stored by other CTAs (generic proxy); the tensor
        // copies read them through the async proxy.
        if (tl.need > 0) ptx::fence_proxy_async_global();
        const size_t kstride = colblock_stride(tl.s_pad);   // every operand has s_pad rows per column block
        const int nh = tl.N >> 1;                                      // this CTA's columns of B
        const uint32_t pair_bytes = 2u * (uint32_t)(kStageBytesA + nh * kBlockK * 2);
        for (int kb = 0; kb < tl.k_blocks; ++kb, ++it) {
          const int s = it % kStages;
          const uint32_t use = it / kStages;
          // stage s is free: the pair MMA has read both CTAs' halves of its last use
          ok = wait_or_abort(ptx::smem_u32(&empty_bar[s]), (use & 1) ^ 1, ab,
                             wait_code(tl.phase, kRoleStageFree));
          if (!ok) break;
          const uint32_t fb_local = ptx::smem_u32(&full_bar[s]);
          const uint32_t fb = ptx::mapa_shared(fb_local, 0);
          if (rank == 0) ptx::mbar_arrive_expect_tx(fb_local, pair_bytes);
          const uint32_t sa = smem_base + (uint32_t)s * kStageBytes, sb = sa + kStageBytesA;
          // two column blocks (K atoms) per stage
          // A: two 16 KB runs, K-major (column blocks 2 kb, 2 kb + 1) or, across
          // the diagonal, MN-major (this CTA's rows as two 64-column blocks).
          const bool at = a_trans(tl, kb), bmn = tl.b_mn || b_trans(tl, kb);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint8_t* asrc = at ? a_block_t(tl, kb, kstride, h) : a_block(tl, 2 * kb + h, kstride);
            ptx::tma_load_2d_pair(sa + (uint32_t)h * 16384u, &tmap_16k, 0, ws_row(p, asrc), fb, pol);
            if (!bmn) {
              const int32_t yb = ws_row(p, b_half_kmajor(tl, 2 * kb + h, kstride, rank));
              if (nh == 128) ptx::tma_load_2d_pair(sb + (uint32_t)h * 16384u, &tmap_16k, 0, yb, fb, pol);
              else ptx::tma_load_2d_pair(sb + (uint32_t)h * 8192u, &tmap_8k, 0, yb, fb, pol);
            }
          }
          if (bmn) {
            // X, or a symmetric B across the diagonal, as the MN-major operand:
            // per 64-column block, the stage's 128 K rows are one contiguous
            // 16 KB run.
            const int per = nh / 64;
            for (int jj = 0; jj < per; ++jj)
              ptx::tma_load_2d_pair(sb + (uint32_t)jj * 16384u, &tmap_16k, 0,
                                    ws_row(p, b_block_mn(tl, 2 * kb, kstride, (int)rank * per + jj)), fb, pol);
          }
        }
      }
      // Drain: the pair MMA has consumed every stage this CTA filled, so no
      // copy into this CTA's shared memory is still in flight (bounded).
      const uint32_t first = it > (uint32_t)kStages ? it - kStages : 0;
      for (uint32_t k = first; k < it; ++k)
        ptx::mbar_wait(ptx::smem_u32(&empty_bar[k % kStages]), (k / kStages) & 1, kWaitLimitNs);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // --------------------------------------------------------- MMA issuer
      // The even CTA issues the pair's MMAs (M = 256: rows 0-127 in its TMEM,
      // 128-255 in the odd CTA's); the odd CTA's issuer only keeps its place
      // in the tile ring.
      uint32_t it = 0, acc_it = 0, seq = 0;
      bool ok = true;
      while (ok) {
        int32_t t;
        if (rank != 0) {
          ok = local_take(ring, seq++, t, ab);
          if (!ok || t >= p.tile_end) break;
          continue;
        }
        ok = local_peek(ring, seq, t, ab);
        if (!ok || t >= p.tile_end) break;
        const Tile tl = ring_tile(ring_tiles, seq);
        // Its operands can only land after the producer's dependency wait;
        // waiting for that first makes a dependency that is never met show up
        // as one (the slot is given back after it, as in the epilogue).
        ok = wait_or_abort(ptx::smem_u32(&dep_bar[seq % kTileRing]), (seq / kTileRing) & 1, ab,
                           wait_code(tl.phase, kRoleDependency));
        local_release(ring, seq);
        ++seq;
        if (!ok) break;
        if (tl.zero || tl.null) continue;
        const uint32_t a = acc_it & 1, ause = acc_it >> 1;
        // both CTAs' epilogues have drained accumulator a
        ok = wait_cluster_or_abort(ptx::smem_u32(&tempty_bar[a]), (ause & 1) ^ 1, ab,
                                   wait_code(tl.phase, kRoleAccFree));
        if (!ok) break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + a * kAccCols;
        for (int kb = 0; kb < tl.k_blocks; ++kb, ++it) {
          const int s = it % kStages;
          const uint32_t use = it / kStages;
          ok = wait_or_abort(ptx::smem_u32(&full_bar[s]), use & 1, ab,
                             wait_code(tl.phase, kRoleStageFull));
          if (!ok) break;
          ptx::tc_fence_after();
          const uint32_t sa = smem_base + (uint32_t)s * kStageBytes, sb = sa + kStageBytesA;
          const uint32_t bh = (uint32_t)(tl.N >> 1) * 128u;   // bytes of one K atom of this CTA's B half
          const bool at = a_trans(tl, kb), bmn = tl.b_mn || b_trans(tl, kb);
          const uint32_t idesc = ptx::idesc_bf16_f32(kPairM, (uint32_t)tl.N, bmn ? 1u : 0u, at ? 1u : 0u);
#pragma unroll
          for (int k = 0; k < kBlockK / 16; ++k) {
            const uint32_t h = (uint32_t)k >> 2, kk = (uint32_t)k & 3;
            // K-major operand: atom h, then 16 elements (32 bytes) inside the
            // swizzle row.  MN-major operand: 16 K rows = two 8-row atoms
            // (2 KB); 64-column blocks 16 KB apart (leading byte offset), 8-row
            // K groups 1 KB apart (stride byte offset).
            const uint64_t adesc = at ? ptx::smem_desc_sw128(sa + (uint32_t)k * 2048u, 16384u, 1024u)
                                      : ptx::smem_desc_sw128(sa + h * 16384u + kk * 32u, 16u, 1024u);
            const uint64_t bdesc = bmn ? ptx::smem_desc_sw128(sb + (uint32_t)k * 2048u, 16384u, 1024u)
                                       : ptx::smem_desc_sw128(sb + h * bh + kk * 32u, 16u, 1024u);
            ptx::umma_bf16_pair(d_tmem, adesc, bdesc, idesc, (kb > 0 || k > 0) ? 1u : 0u);
          }
          // frees stage s in both CTAs once these MMAs have read it
          ptx::umma_commit_pair_multicast(ptx::smem_u32(&empty_bar[s]), kPair);
        }
        if (!ok) break;
        ptx::umma_commit_pair_multicast(ptx::smem_u32(&tfull_bar[a]), kPair);   // both CTAs' accumulators complete
        ++acc_it;
      }
      if (rank == 0) {
        // Every MMA this thread issued has completed (and its commits have
        // arrived) before TMEM is released.
        ptx::umma_commit_pair_multicast(ptx::smem_u32(&drain_bar), 0x1);
        ptx::mbar_wait(ptx::smem_u32(&drain_bar), 0, kWaitLimitNs);
      }
    }
    __syncwarp();
  } else if (warp < kSchedulerWarp) {
    // -------------------------------------------------------------- epilogue
    // Eight warps: warp w reads TMEM lane quadrant w % 4 (the hardware rule)
    // and one half of the tile's columns.  Every wait's outcome is made
    // warp-uniform before the warp acts on it (tcgen05.ld is warp-wide).
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    const int k = (warp - 2 - 4 * half) * 32 + lane;   // this thread within its half (0..127)
    uint8_t* const stage = smem_raw + ((smem_base + (uint32_t)kStages * kStageBytes) - ptx::smem_u32(smem_raw)) +
                           (size_t)half * kStageOutBytes;
    const uint32_t hbar = ptx::smem_u32(&half_bar[half]);
    uint32_t hphase = 0;
    uint32_t acc_it = 0, seq = 0;
    bool live = true;
    while (live) {
      int32_t t = 0;
      int got_tile = 1;
      if (lane == 0) got_tile = local_peek(ring, seq, t, ab);
      t = __shfl_sync(0xffffffffu, t, 0);
      if (!__shfl_sync(0xffffffffu, got_tile, 0) || t >= p.tile_end) break;
      const Tile tl = ring_tile(ring_tiles, seq);
      __syncwarp();   // every lane has its copy before lane 0 gives the slot back
      // The tile's earlier products are stored (this CTA's producer has seen
      // them, dep_bar) before its epilogue input is read; the ring slot is
      // given back only after this wait, so dep_bar's phases cannot run ahead
      // of it.
      if (lane == 0) {
        got_tile = wait_or_abort(ptx::smem_u32(&dep_bar[seq % kTileRing]), (seq / kTileRing) & 1, ab,
                                 wait_code(tl.phase, kRoleDependency));
        local_release(ring, seq);
      }
      ++seq;
      if (!__shfl_sync(0xffffffffu, got_tile, 0)) break;
      const NsMat& d = p.mat[tl.mi];
      const int rrow = quad * 32 + lane;                 // this thread's row of the CTA's 128
      const int m = tl.mc + rrow;                        // its output row
      const int cw = tl.N >> 1;                          // columns of this half (128, or 64)
      const int c0 = half * cw;
      if (tl.zero || tl.null) {
        if (tl.zero && (tl.mode == kUpdateFinal || tl.mode == kFinalQ)) {
          float z[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) z[j] = 0.f;
          for (int c = c0; c < c0 + cw; c += 32) store_final(d, p, m, tl.n0 + c, z);
        }
        continue;
      }
      const size_t stride = colblock_stride(d.s_pad);
      const bool has_c = tl.c_in != nullptr;
      const bool final_out = tl.mode == kUpdateFinal || tl.mode == kFinalQ;
      // a tall matrix's final update writes through the stage transposed (the
      // standard form's epilogue input, X, is first read out of the stage
      // into registers, block by block)
      const bool final_t = final_out && d.transposed && d.vec_ok && d.out != nullptr && d.w == nullptr;
      const int nblk = cw >> 6;                          // 64-column blocks of this half
      const size_t run_off = (size_t)(tl.mc >> 3) * 1024;   // the CTA's rows in a column block
      // The epilogue input (A or X) does not depend on the accumulator: fetch
      // the first block before waiting for the MMAs, the next while the
      // current one is processed.
      uint4 pre[kRunChunks];
      if (has_c) load_run(tl.c_in + (size_t)((tl.n0 + c0) >> 6) * stride + run_off, k, pre);
      const float2 nrm = p.norm[d.norm_idx];             // read before the wait too: its latency hides under it
      const uint32_t a = acc_it & 1, ause = acc_it >> 1;
      const bool got = wait_or_abort(ptx::smem_u32(&tfull_bar[a]), ause & 1, ab,
                                     wait_code(tl.phase, kRoleAccFull));
      if (!__all_sync(0xffffffffu, got)) break;
      ptx::tc_fence_after();
      const float scale_gram = tl.first ? nrm.y * nrm.y : 1.0f;
      const float scale_upd = (tl.first || tl.mode == kFinalQ) ? nrm.y : 1.0f;
      const uint32_t t_row = tmem_base + a * kAccCols + ((uint32_t)(quad * 32) << 16);
      const int32_t code = wait_code(tl.phase, kRoleAccFull);
      if (final_t) {
        // A tall matrix's final update, through the stage transposed: per
        // 64-column block, the epilogue input (X, standard form) is staged and
        // each row's 64 values read back into registers; then per 32-column
        // chunk the outputs are staged transposed and copied out.
        for (int blk = 0; blk < nblk && live; ++blk) {
          const int nb = tl.n0 + c0 + 64 * blk;          // first column of this 64-column block
          if (has_c) {
            if (blk > 0) load_run(tl.c_in + (size_t)(nb >> 6) * stride + run_off, k, pre);
            put_run(stage, k, pre);
            if (!half_sync(hbar, hphase, ab, code)) { live = false; break; }   // the input block is staged
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              pre[q] = *reinterpret_cast<const uint4*>(stage + stage_off(rrow, 0, q));
              pre[4 + q] = *reinterpret_cast<const uint4*>(stage + stage_off(rrow, 32, q));
            }
            if (!half_sync(hbar, hphase, ab, code)) { live = false; break; }   // the stage takes the outputs
          }
#pragma unroll 1
          for (int hc = 0; hc < 2; ++hc) {
            const int cb = 32 * hc;                      // columns [cb, cb + 32) of the block
            uint32_t r[32];
            ptx::tmem_ld_32x32b_x32(t_row + (uint32_t)(nb - tl.n0 + cb), r);
            ptx::tmem_ld_wait();
            if (blk == nblk - 1 && hc == 1) {
              // last accumulator read: hand it back to the MMA warp
              ptx::tc_fence_before();
              __syncwarp();
              if (lane == 0) ptx::mbar_arrive_signal(ptx::mapa_shared(ptx::smem_u32(&tempty_bar[a]), 0));
            }
            float v[32];
            if (has_c) {
              uint4 xin[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) xin[q] = hc == 0 ? pre[q] : pre[4 + q];
              float x[32];
              unpack_bf16x32(xin, x);
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = fmaf(p.a, x[j], __uint_as_float(r[j])) * scale_upd;
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]) * scale_upd;
            }
            stage_final_t(stage, rrow, v, p.out_bf16 != 0);
            if (!half_sync(hbar, hphase, ab, code)) { live = false; break; }   // the chunk is staged
            store_final_t(d, p, stage, tl.mc, nb + cb, k);
            if (!half_sync(hbar, hphase, ab, code)) { live = false; break; }   // and copied out
          }
        }
      } else {
        for (int blk = 0; blk < nblk && live; ++blk) {
          const int nb = tl.n0 + c0 + 64 * blk;            // first column of this 64-column block
          // Symmetric products write their tiles as they are: the blocks below
          // the diagonal of 256 x 256 blocks are never stored (the products that
          // read them read the stored blocks across it, transposed).
          const bool staged_out = !final_out;
          if (has_c) {
            put_run(stage, k, pre);
            if (!half_sync(hbar, hphase, ab, code)) { live = false; break; }   // the input block is staged
            if (blk + 1 < nblk) load_run(tl.c_in + (size_t)((nb + 64) >> 6) * stride + run_off, k, pre);
          }
#pragma unroll 1
          for (int hc = 0; hc < 2; ++hc) {
            const int cb = 32 * hc;                        // columns [cb, cb + 32) of the block
            // this row's input chunk, read from the stage before the TMEM read
            // so that the two latencies overlap
            uint4 xin[4];
            if (has_c) {
#pragma unroll
              for (int q = 0; q < 4; ++q) xin[q] = *reinterpret_cast<const uint4*>(stage + stage_off(rrow, cb, q));
            }
            uint32_t r[32];
            ptx::tmem_ld_32x32b_x32(t_row + (uint32_t)(nb - tl.n0 + cb), r);
            ptx::tmem_ld_wait();
            if (blk == nblk - 1 && hc == 1) {
              // last accumulator read: hand it back to the MMA warp (the even
              // CTA's barrier; the signal carries no data, see mbar_arrive_signal)
              ptx::tc_fence_before();
              __syncwarp();
              if (lane == 0) ptx::mbar_arrive_signal(ptx::mapa_shared(ptx::smem_u32(&tempty_bar[a]), 0));
            }
            float v[32];
            if (tl.mode == kGram) {
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]) * scale_gram;
            } else if (tl.mode == kFinalQ) {
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]) * scale_upd;
            } else {
              float x[32];
              unpack_bf16x32(xin, x);
              if (tl.mode == kPoly || tl.mode == kPolyI) {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = fmaf(p.c, __uint_as_float(r[j]), p.b * x[j]);
                if (tl.mode == kPolyI) {
                  // a I: the diagonal element of this row, if among these columns
#pragma unroll
                  for (int j = 0; j < 32; ++j)
                    if (nb + cb + j == m) v[j] += p.a;
                }
              } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = fmaf(p.a, x[j], __uint_as_float(r[j])) * scale_upd;
              }
            }
            const int n = nb + cb;
            if (final_out) store_final(d, p, m, n, v);
            else stage_chunk(stage, rrow, cb, v);
          }
          if (staged_out) {
            if (!half_sync(hbar, hphase, ab, code)) { live = false; break; }   // the output block is staged
            store_run(static_cast<uint8_t*>(tl.out) + (size_t)(nb >> 6) * stride + run_off, stage, k);
          }
          // the stage is free again before anyone writes the next block into it
          // (after the last block: once this warp's share is published)
          if (blk + 1 < nblk && !half_sync(hbar, hphase, ab, code)) { live = false; break; }
        }
      }
      if (!live) break;
      ++acc_it;
      if (!tl.last) {
        // Publish this warp's share of the tile: every lane's stores are
        // ordered before the tensor copies that later tiles issue after
        // reading the counter (proxy fence), and before lane 0's release add
        // (the warp barrier orders the lanes' stores before it; the release is
        // cumulative over them).
        ptx::fence_proxy_async_global();
        __syncwarp();
        if (lane == 0) ptx::red_release_gpu_add(p.done + tl.mi, 1);
      }
      // ... and before anyone writes the next tile into it
      if (!half_sync(hbar, hphase, ab, wait_code(tl.phase, kRoleAccFull))) break;
    }
  } else {
    if (lane == 0) {
      // ----------------------------------------------------------- scheduler
      // Even CTA: takes the pair's tiles in list order, marks each "ready"
      // or "wait" from one read of its matrix's counter, and hands it to this
      // CTA's roles and to the odd CTA's scheduler (the end marker last); it
      // takes the next tile only once this one may start (below), so a pair
      // that cannot start a tile takes no more of the list, which other pairs
      // may be able to start.  Odd CTA: forwards what it receives to its own
      // roles, then frees the pair slot.  Each hand-over across the pair costs
      // a cluster-scope release (~850 cycles), which is why the producers wait
      // for the dependencies themselves and the local hand-overs go first.
      uint32_t seq = 0;
      while (true) {
        int32_t t;
        if (rank == 0) {
          t = p.tile_begin + atomicAdd(p.next_tile, 1);
          if (t > p.tile_end) t = p.tile_end;           // the end marker
          bool ready = true;
          Tile tl{}, tl_odd{};
          if (t < p.tile_end) {
            tl = decode_tile(p, t, 0);
            tl_odd = tl;
            tl_odd.mc += kBlockM;                          // the odd CTA's rows (all that differs)
            const int32_t need = t == p.stall_tile ? INT32_MAX : tl.need;   // the test hook: a count never reached
            ready = tl.zero || tl.null || need <= 0 || ptx::ld_acquire_gpu(p.done + tl.mi) >= need;
          }
          const int32_t v = ready ? t : (t | kPollBit);
          const bool last = t >= p.tile_end;
          if (!local_publish(ring, seq, v, ab, ring_tiles, last ? nullptr : &tl) ||
              !pair_publish(pair, seq, v, ab, ptx::smem_u32(&pair_tiles[0]), last ? nullptr : &tl_odd))
            break;
          // A pair takes its next tile only once this one may start.  In a
          // launch with many tiles the scheduler watches the counter itself
          // and moves on as soon as the tile is ready, so the few tiles it has
          // taken ahead keep the pair busy across a wait.  In a launch with
          // few tiles per iteration (narrow tiles) a pair takes one tile at a
          // time, waiting until its producer has passed the dependency: one
          // holding several would run them one after another while other
          // pairs sit idle at the end of the product.
          if (t < p.tile_end) {
            if (p.narrow) {
              if (!wait_or_abort(ptx::smem_u32(&dep_bar[seq % kTileRing]), (seq / kTileRing) & 1, ab,
                                 wait_code(0, kRoleDependency)))
                break;
            } else if (!ready) {
              const int32_t need = t == p.stall_tile ? INT32_MAX : tl.need;
              if (!wait_done(p.done + tl.mi, need, ab, wait_code(tl.phase, kRoleDependency))) break;
            }
          }
        } else {
          if (!pair_take(pair, seq, t, ab)) break;
          const bool last = (t & ~kPollBit) >= p.tile_end;
          if (!local_publish(ring, seq, t, ab, ring_tiles, last ? nullptr : &pair_tiles[seq % kPairRing])) break;
          pair_free(pair, seq);
          t &= ~kPollBit;
        }
        ++seq;
        if (t >= p.tile_end) break;
      }
    }
    __syncwarp();
  }

  // Teardown: no CTA of the pair leaves (or frees TMEM) while its peer may
  // still multicast into its shared memory or arrive on its barriers.
  ptx::tc_fence_before();
  ptx::cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

}  // namespace

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The CUDA driver API's tensor-map encoder, looked up once through the
// runtime (the library links no driver library).
EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// CTA pairs of ns_kernel that fit on the device at once (one CTA per SM),
// worked out once per device: the kernel is persistent and the grid is this
// many pairs (or fewer, for a short tile list).
cudaError_t resident_pairs(int dev, int* out) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static int pairs[kMaxDevices] = {};
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (pairs[dev] == 0) {
    cudaError_t e = cudaFuncSetAttribute(ns_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGemmSmemBytes);
    if (e != cudaSuccess) return e;
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * (sms / 2)), 1, 1);
    cfg.blockDim = dim3(kGemmThreads, 1, 1);
    cfg.dynamicSmemBytes = kGemmSmemBytes;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, ns_kernel, &cfg);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    pairs[dev] = n;
  }
  *out = pairs[dev];
  return cudaSuccess;
}

// The wait limit of one launch.  The longest legitimate wait is a tile's
// wait for the earlier products of its matrix (and its pair's roles waiting
// behind it for the tile): those products sit before it in the product-major
// tile list, so it ends once the machine has worked through at most one whole
// product of every matrix of the launch.  The limit is 8x the largest such
// product's executed FLOPs at a conservative rate -- every CTA pair at a
// quarter of its tensor peak of 16384 bf16 FLOP per clock, at 1 GHz -- and
// never below 2 s (nor above an hour).  Only a launch whose largest product
// would take more than 0.25 s at that rate (~35 ms at full speed; short sides
// in the tens of thousands) gets more than 2 s: the 8B owner set's largest
// product, 6.9 TFLOP, takes 22 ms at that rate.
uint64_t wait_limit_ns(const NsBatch& b, int pairs) {
  double prod[3] = {0.0, 0.0, 0.0};
  for (int i = 0; i < b.n; ++i) {
    const NsMat& d = b.mat[i];
    const double tile = 2.0 * kPairM * ((b.narrow_mask >> kGram) & 1 ? kBlockN / 2 : kBlockN);   // FLOPs of one symmetric tile per unit of K
    prod[kGram] += d.tiles_sym * tile * d.l_pad;
    prod[kPoly] += d.tiles_sym * tile * d.s_pad;
    prod[kUpdate] += 2.0 * d.s_pad * (double)d.s_pad * d.l_pad;
  }
  const double worst = prod[0] > prod[1] ? (prod[0] > prod[2] ? prod[0] : prod[2]) : (prod[1] > prod[2] ? prod[1] : prod[2]);
  const double rate = (double)(pairs > 0 ? pairs : 1) * 16384.0 * 0.25 * 1e9;   // FLOP/s
  double ns = 8.0 * worst / rate * 1e9;
  if (ns < (double)kWaitLimitNs) ns = (double)kWaitLimitNs;
  if (ns > 3.6e12) ns = 3.6e12;
  return (uint64_t)ns;
}

}  // namespace

// The whole workspace as a 2-D tensor of 128-byte rows, with two boxes: 128
// rows (16 KB: a CTA's A rows or K-major B half) and 64 rows (8 KB: one
// column block of the MN-major X, or a 64-column B half).  Every operand run of
// the blocked layout starts on a row and lands in shared memory byte for byte
// (no swizzle: the layout is already in UMMA's 128-byte-swizzle order).  Fewer,
// larger copies keep the pair fed: with 8 KB copies throughout the pipeline
// ran about 11 % slower.
cudaError_t launch_ns(const NsBatch& b, size_t ws_bytes, cudaStream_t s) {
  const int total_tiles = b.tile_end - b.tile_begin;
  if (total_tiles <= 0) return cudaSuccess;
  const EncodeTiledFn encode = encode_fn();
  if (!encode) return cudaErrorNotSupported;
  CUtensorMap tmap_8k, tmap_16k;
  const cuuint64_t dims[2] = {128, (cuuint64_t)(ws_bytes / 128)};
  const cuuint64_t strides[1] = {128};
  const cuuint32_t box_8k[2] = {128, 64};
  const cuuint32_t box_16k[2] = {128, 128};
  const cuuint32_t estride[2] = {1, 1};
  if (encode(&tmap_8k, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(b.ws), dims, strides, box_8k, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  if (encode(&tmap_16k, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(b.ws), dims, strides, box_16k, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int max_clusters = 0;
  e = resident_pairs(dev, &max_clusters);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = kGemmSmemBytes;
  cfg.stream = s;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  const int clusters = total_tiles < max_clusters ? total_tiles : max_clusters;
  cfg.gridDim = dim3((unsigned)(2 * clusters), 1, 1);
  NsBatch lb = b;
  lb.wait_limit_ns = wait_limit_ns(b, clusters);
  e = cudaLaunchKernelEx(&cfg, ns_kernel, lb, tmap_8k, tmap_16k);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mfsdp
