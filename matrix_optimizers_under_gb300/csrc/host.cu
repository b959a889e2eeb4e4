// Host side of the C ABI: argument checks, workspace layout, and the launch
// sequence of the owner-local optimizer step.
//
// MatrixFSDP: Communication-Free Matrix Optimizers Under ZeRO-3 Parameter
// Sharding -- Abstract: the owner rank holds each owned matrix whole in its
// owner shard (MatrixShard metadata: offset, rows, cols), applies Muon
// momentum and Newton-Schulz locally, and applies AdamW to the packed tail.
//
// Launch sequence of mfsdp_muon_owner_step on one stream:
//   momentum/segment-view kernel (grouped over all shards)
//   norm finalise
//   ns_steps x { Gram, polynomial, update }   (one persistent launch)
// Grouped launches carry their per-matrix table as a kernel parameter, at most
// kMaxBatch matrices per launch.
#include <algorithm>
#include <climits>
#include <cmath>
#include <cstring>
#include <atomic>
#include <mutex>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "mfsdp.h"
#include "mfsdp_internal.h"

namespace mfsdp {
namespace {

constexpr size_t kHeaderBytes = 256;

// NVTX range around the host-side queuing of one phase (visible to nsys, and
// to ncu's --nvtx-include filters; free when no tool is attached).
struct PhaseRange {
  explicit PhaseRange(const char* name) { nvtxRangePushA(name); }
  ~PhaseRange() { nvtxRangePop(); }
  PhaseRange(const PhaseRange&) = delete;
  PhaseRange& operator=(const PhaseRange&) = delete;
};

// Test hook (mfsdp_test_inject_stall): the tile whose dependency wait the next
// Newton-Schulz launch makes unreachable, -1 for none.  One-shot.
std::atomic<int32_t> g_stall_tile{-1};

// Copy streams and events of the host-buffer step, per device.
constexpr int kMaxPipeDevices = 64;
struct CopyPipe {
  std::mutex mu;
  cudaStream_t s_in = nullptr, s_out = nullptr;
  std::vector<cudaEvent_t> ev;
};
CopyPipe g_pipe[kMaxPipeDevices];

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct MatLayout {
  int s, l, s_pad, l_pad;
  int transposed;
  int gram_ok;           // the shape may run the Gram-space program (gram_space_shape)
  size_t x0, x1, a, b;   // byte offsets in the workspace
  size_t c, q0, q1;      // Gram-space program: C and the Q ping-pong, inside X1's region
  int tiles_k1;          // momentum-kernel tiles (kTile x kTile over s_pad x l_pad)
  int partial0;
};

struct Layout {
  std::vector<MatLayout> mats;
  size_t norm_off = 0;
  size_t done_off = 0;     // Newton-Schulz tile counter, then one completion counter per matrix
  size_t partial_off = 0;
  int partials = 0;
  size_t bytes = 0;
};

int shape_ok(const mfsdp_matrix_shard& sh) {
  if (sh.rows < 1 || sh.cols < 1) return MFSDP_ERR_UNSUPPORTED_SHAPE;
  const int64_t s = std::min(sh.rows, sh.cols), l = std::max(sh.rows, sh.cols);
  if (s > MFSDP_MAX_SHORT_SIDE || l > MFSDP_MAX_LONG_SIDE) return MFSDP_ERR_UNSUPPORTED_SHAPE;
  return MFSDP_OK;
}

// Shapes that run the Gram-space program (for 1 .. kGramSpaceMaxSteps steps):
// a long side at least twice the short side, where it executes about half
// the standard program's tensor FLOPs and keeps the long K = l out of every
// iteration but the first, and a short side of at least 128.  A bf16
// emulation of both programs against the fp64 definition gives the
// Gram-space one the same or a smaller relative error on such shapes (0.7-1.1 %
// at 5 steps), and a larger one on near-square shapes (5 % at l = s), which
// keep the standard program.  Below a short side of 384 the long side must
// also exceed it by 384: the Gram-space program runs one product more, which
// on a small latency-bound matrix costs more than its shorter Gram products
// save (256 x 512 alone: 1.03x the time).
int gram_space_shape(int s, int l) { return s >= 128 && l >= 2 * s && l >= s + 384; }

bool use_gram_space(const MatLayout& m, int32_t ns_steps) {
  return m.gram_ok && ns_steps >= 1 && ns_steps <= kGramSpaceMaxSteps;
}

int make_layout(const mfsdp_matrix_shard* shards, int n, Layout* L) {
  if (n < 0 || (n > 0 && !shards)) return MFSDP_ERR_INVALID_ARG;
  L->mats.resize(n);
  int partials = 0;
  for (int i = 0; i < n; ++i) {
    const int st = shape_ok(shards[i]);
    if (st != MFSDP_OK) return st;
    MatLayout& m = L->mats[i];
    m.s = (int)std::min(shards[i].rows, shards[i].cols);
    m.l = (int)std::max(shards[i].rows, shards[i].cols);
    m.s_pad = (int)round_up((size_t)m.s, kPadS);
    m.l_pad = (int)round_up((size_t)m.l, kPad);
    m.transposed = shards[i].rows > shards[i].cols ? 1 : 0;
    m.gram_ok = gram_space_shape(m.s, m.l);
    m.tiles_k1 = (m.s_pad / kTile) * (m.l_pad / kTile);
    m.partial0 = partials;
    partials += m.tiles_k1;
  }
  size_t off = kHeaderBytes;
  L->norm_off = off;
  off = round_up(off + sizeof(float2) * (size_t)n, 256);
  L->done_off = off;
  off = round_up(off + sizeof(int32_t) * (size_t)(n + 1), 256);
  L->partial_off = off;
  L->partials = partials * kPartialsPerTile;
  off = round_up(off + sizeof(float) * (size_t)L->partials, 1024);
  for (int i = 0; i < n; ++i) {
    MatLayout& m = L->mats[i];
    const size_t xb = (size_t)m.s_pad * m.l_pad * 2, ab = (size_t)m.s_pad * m.s_pad * 2;
    m.x0 = off; off += xb;
    // X1 (standard program) or C and the two Q (Gram-space program)
    m.x1 = off;
    m.c = off;
    m.q0 = off + ab;
    m.q1 = off + 2 * ab;
    off += m.gram_ok ? std::max(xb, 3 * ab) : xb;
    m.a = off; off += ab;
    m.b = off; off += ab;
  }
  L->bytes = off;
  return MFSDP_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool ranges_overlap(const void* p, size_t pb, const void* q, size_t qb) {
  if (pb == 0 || qb == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(p), b0 = reinterpret_cast<uintptr_t>(q);
  return a0 < b0 + qb && b0 < a0 + pb;
}

size_t dtype_size(int32_t dt) { return dt == MFSDP_DTYPE_BF16 ? 2 : 4; }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MFSDP_OK : MFSDP_ERR_CUDA; }

// The workspace header holds the device status word; an entry point clears it
// once, before its first kernel, so a failure anywhere in the call stays
// visible to mfsdp_muon_device_status.
int clear_status(uint8_t* ws, cudaStream_t stream) { return cuda_status(cudaMemsetAsync(ws, 0, kHeaderBytes, stream)); }

// Output tiling of one product of one matrix, in tiles of the 256 rows a CTA
// pair computes together and `width` (256, or 128 for narrow tiles) columns.
// The Gram and polynomial outputs are symmetric: only the tiles on or above
// the diagonal of 256 x 256 blocks are computed (for narrow tiles: the two
// 128-column halves of each) and stored; the products that read them read the
// blocks below that diagonal from their stored transposes.
struct GemmTiling {
  int tiles, tiles_m, tiles_n, n_last, symmetric;
};

GemmTiling gemm_tiling(int mode, int s_pad, int l_pad, int width = kBlockN) {
  GemmTiling t;
  t.tiles_m = s_pad / kPairM;
  if (mode == kGram || mode == kPoly) {
    const int nb2 = s_pad / kPairM;
    t.symmetric = 1;
    t.tiles_n = nb2 * (kBlockN / width);
    t.n_last = width;
    t.tiles = nb2 * (nb2 + 1) / 2 * (kBlockN / width);
  } else {
    t.symmetric = 0;
    t.tiles_n = (l_pad + width - 1) / width;
    t.n_last = l_pad - (t.tiles_n - 1) * width;
    t.tiles = t.tiles_m * t.tiles_n;
  }
  return t;
}

// Tile widths of a launch.  A launch whose tiles per Newton-Schulz iteration
// at the full width are fewer than twice the SMs is "narrow": such an owner
// set is bound by its chain of dependent products.  In it, a product whose
// full-width tiles are fewer than the CTA pairs (half the SMs) uses narrow
// tiles (256 x 128): twice the tiles for the idle pairs, half the epilogue
// each, on the chain; a product with more tiles keeps the full width, since a
// narrow pair MMA runs at half the full-width rate and such a product is
// bound by its pairs' throughput.  Larger sets keep the full width
// throughout.  Every output element sums its products in the same order at
// either width, so the update is bit for bit the same.  Returns the launch's
// flag; *mask (bit k: product k narrow) receives the widths.
bool use_narrow_tiles(const Layout& L, int base, int cnt, int32_t* mask) {
  *mask = 0;
  static std::mutex mu;
  static int sms[kMaxPipeDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxPipeDevices) return false;
  int n_sm = 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (sms[dev] == 0 && cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      sms[dev] = 0;
    n_sm = sms[dev];
  }
  if (n_sm <= 0) return false;
  int64_t sym = 0, upd = 0;
  for (int i = base; i < base + cnt; ++i) {
    const MatLayout& m = L.mats[i];
    sym += gemm_tiling(kGram, m.s_pad, m.l_pad).tiles;
    upd += gemm_tiling(kUpdate, m.s_pad, m.l_pad).tiles;
  }
  if (2 * sym + upd >= 2 * (int64_t)n_sm) return false;
  if (2 * sym < n_sm) *mask |= (1 << kGram) | (1 << kPoly);
  if (2 * upd < n_sm) *mask |= 1 << kUpdate;
  return true;
}

// Tensor-core FLOPs one product of one matrix executes: outputs padded to
// 256 (short side) and 128 (long side), symmetric products on their 256 x 256
// pair tiles on or above the diagonal; a contraction over the short side runs
// to s rounded up to 128 (the K loop skips the all-zero padding beyond it).
uint64_t executed_flops(int mode, int s, int s_pad, int l_pad) {
  const uint64_t nb2 = (uint64_t)s_pad / kPairM;
  const uint64_t tile = (uint64_t)kPairM * kPairM * 2;
  const uint64_t k_s = (uint64_t)round_up((size_t)s, kBlockK);
  if (mode == kGram) return nb2 * (nb2 + 1) / 2 * tile * (uint64_t)l_pad;
  if (mode == kPoly) return nb2 * (nb2 + 1) / 2 * tile * k_s;
  return 2ull * s_pad * (uint64_t)l_pad * k_s;
}

// The Newton-Schulz launch indexes its tiles and counts completions in int32:
// a batch's tiles over all iterations, and one matrix's completion count
// (2 * kEpilogueWarps per tile), must fit.
bool ns_counts_fit(const Layout& L, int32_t ns_steps) {
  const int n = (int)L.mats.size();
  for (int base = 0; base < n; base += kMaxBatch) {
    int64_t batch = 0, fin = 0;
    for (int i = base; i < std::min(n, base + kMaxBatch); ++i) {
      const MatLayout& m = L.mats[i];
      // narrow tiles, the larger count; either program (the Gram-space one
      // has four symmetric products per iteration and a final update-like one)
      const int64_t sym = gemm_tiling(kGram, m.s_pad, m.l_pad, kBlockN / 2).tiles;
      const int64_t upd = gemm_tiling(kUpdate, m.s_pad, m.l_pad, kBlockN / 2).tiles;
      const int64_t per_iter = 4 * sym + upd;
      if ((per_iter * ns_steps + upd) * 2 * kEpilogueWarps > INT32_MAX) return false;
      batch += per_iter;
      fin += upd;
    }
    // headroom: pairs overshoot the tile counter; bit 30 of a handed-out
    // tile index is a flag
    if (batch * ns_steps + fin > (int64_t(1) << 30) - 65536) return false;
  }
  return true;
}

int launch_momentum_phase(const mfsdp_matrix_shard* shards, int n_shards, const Layout& L, const void* grad,
                          int32_t grad_dtype, float* momentum, float beta, int32_t nesterov, float eps, uint8_t* ws,
                          cudaStream_t stream);
// Optional last-epilogue application of the update to the weights.
struct ApplyArgs {
  void* w;            // flat weights, same offsets as the gradient
  int32_t w_dtype;
  double lr, wd;
  int32_t scale_mode; // 0: 1; 1: sqrt(max(1, rows/cols)); 2: 0.2*sqrt(max(rows, cols))
};

int launch_ns_phase(const mfsdp_matrix_shard* shards, int n_shards, const Layout& L, void* update,
                    int32_t update_dtype, int32_t ns_steps, float a, float b, float c, uint8_t* ws,
                    cudaStream_t stream, const ApplyArgs* apply = nullptr);

double shape_scale(int64_t rows, int64_t cols, int32_t mode) {
  if (mode == 1) return std::sqrt(std::max(1.0, (double)rows / (double)cols));
  if (mode == 2) return 0.2 * std::sqrt((double)std::max(rows, cols));
  return 1.0;
}

}  // namespace
}  // namespace mfsdp

using namespace mfsdp;

extern "C" const char* mfsdp_status_string(int status) {
  switch (status) {
    case MFSDP_OK: return "ok";
    case MFSDP_ERR_INVALID_ARG: return "invalid argument";
    case MFSDP_ERR_MISALIGNED: return "misaligned pointer";
    case MFSDP_ERR_OVERLAP: return "overlapping segments or buffers";
    case MFSDP_ERR_OUT_OF_BOUNDS: return "segment out of bounds";
    case MFSDP_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype";
    case MFSDP_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MFSDP_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MFSDP_ERR_CUDA: return "CUDA runtime error";
    case MFSDP_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case MFSDP_ERR_IO: return "checkpoint file input/output error";
    case MFSDP_ERR_FORMAT: return "not a valid checkpoint file";
    default: return "unknown status";
  }
}

extern "C" const char* mfsdp_version(void) { return "0.10.5"; }

extern "C" size_t mfsdp_muon_workspace_bytes(const mfsdp_matrix_shard* shards, int32_t n_shards) {
  Layout L;
  if (make_layout(shards, n_shards, &L) != MFSDP_OK) return 0;
  return L.bytes;
}

extern "C" int mfsdp_muon_workspace_layout(const mfsdp_matrix_shard* shards, int32_t n_shards, int64_t* out) {
  Layout L;
  const int st = make_layout(shards, n_shards, &L);
  if (st != MFSDP_OK) return st;
  if (n_shards > 0 && !out) return MFSDP_ERR_INVALID_ARG;
  for (int i = 0; i < n_shards; ++i) {
    const MatLayout& m = L.mats[i];
    int64_t* o = out + 8 * i;
    o[0] = (int64_t)m.x0; o[1] = (int64_t)m.x1; o[2] = (int64_t)m.a; o[3] = (int64_t)m.b;
    o[4] = m.s_pad; o[5] = m.l_pad; o[6] = m.s; o[7] = m.l;
  }
  return MFSDP_OK;
}

namespace mfsdp {
namespace {

// Every check of an owner step's arguments that needs no workspace (host only,
// nothing queued).
int validate_step_args(const mfsdp_matrix_shard* shards, int32_t n_shards, const void* grad, int32_t grad_dtype,
                       const float* momentum, const void* update, int32_t update_dtype, int64_t numel, double beta,
                       int32_t nesterov, int32_t ns_steps, double a, double b, double c, double eps, Layout* L) {
  if (n_shards < 0 || (n_shards > 0 && !shards)) return MFSDP_ERR_INVALID_ARG;
  if (!std::isfinite(beta) || !std::isfinite(a) || !std::isfinite(b) || !std::isfinite(c) || !std::isfinite(eps) ||
      eps < 0.0)
    return MFSDP_ERR_INVALID_ARG;
  if (grad_dtype != MFSDP_DTYPE_F32 && grad_dtype != MFSDP_DTYPE_BF16) return MFSDP_ERR_UNSUPPORTED_DTYPE;
  if (update_dtype != MFSDP_DTYPE_F32 && update_dtype != MFSDP_DTYPE_BF16) return MFSDP_ERR_UNSUPPORTED_DTYPE;
  if (numel < 0 || ns_steps < 0 || ns_steps > 64 || (nesterov != 0 && nesterov != 1)) return MFSDP_ERR_INVALID_ARG;
  if (n_shards == 0) return MFSDP_OK;
  if (!grad || !momentum || !update) return MFSDP_ERR_INVALID_ARG;
  if (!aligned(grad, 16) || !aligned(momentum, 16) || !aligned(update, 16)) return MFSDP_ERR_MISALIGNED;
  const int st = make_layout(shards, n_shards, L);
  if (st != MFSDP_OK) return st;
  if (!ns_counts_fit(*L, ns_steps)) return MFSDP_ERR_UNSUPPORTED_SHAPE;
  // The Newton-Schulz tensor copies address the workspace in 128-byte rows
  // with int32 coordinates.
  if (L->bytes / 128 >= (size_t)INT32_MAX) return MFSDP_ERR_UNSUPPORTED_SHAPE;
  for (int i = 0; i < n_shards; ++i) {
    const mfsdp_matrix_shard& sh = shards[i];
    if (sh.offset < 0 || sh.offset > numel || sh.rows * sh.cols > numel - sh.offset) return MFSDP_ERR_OUT_OF_BOUNDS;
  }
  std::vector<int> ord(n_shards);
  for (int i = 0; i < n_shards; ++i) ord[i] = i;
  std::sort(ord.begin(), ord.end(), [&](int x, int y) { return shards[x].offset < shards[y].offset; });
  for (int k = 1; k < n_shards; ++k) {
    const mfsdp_matrix_shard& p0 = shards[ord[k - 1]];
    if (p0.offset + p0.rows * p0.cols > shards[ord[k]].offset) return MFSDP_ERR_OVERLAP;
  }
  const size_t gbytes = (size_t)numel * dtype_size(grad_dtype), mbytes = (size_t)numel * 4,
               ubytes = (size_t)numel * dtype_size(update_dtype);
  const bool in_place = (update == grad && update_dtype == grad_dtype);
  if (ranges_overlap(momentum, mbytes, grad, gbytes) || ranges_overlap(momentum, mbytes, update, ubytes) ||
      (!in_place && ranges_overlap(grad, gbytes, update, ubytes)))
    return MFSDP_ERR_OVERLAP;
  return MFSDP_OK;
}

// validate_step_args, then the workspace: present, aligned, large enough and
// apart from the other buffers.
int validate_step(const mfsdp_matrix_shard* shards, int32_t n_shards, const void* grad, int32_t grad_dtype,
                  const float* momentum, const void* update, int32_t update_dtype, int64_t numel, double beta,
                  int32_t nesterov, int32_t ns_steps, double a, double b, double c, double eps,
                  const void* workspace, size_t workspace_bytes, Layout* L) {
  const int st = validate_step_args(shards, n_shards, grad, grad_dtype, momentum, update, update_dtype, numel, beta,
                                    nesterov, ns_steps, a, b, c, eps, L);
  if (st != MFSDP_OK || n_shards == 0) return st;
  if (!workspace) return MFSDP_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return MFSDP_ERR_MISALIGNED;
  if (workspace_bytes < L->bytes) return MFSDP_ERR_WORKSPACE_TOO_SMALL;
  const size_t gbytes = (size_t)numel * dtype_size(grad_dtype), mbytes = (size_t)numel * 4,
               ubytes = (size_t)numel * dtype_size(update_dtype);
  if (ranges_overlap(workspace, L->bytes, grad, gbytes) || ranges_overlap(workspace, L->bytes, momentum, mbytes) ||
      ranges_overlap(workspace, L->bytes, update, ubytes))
    return MFSDP_ERR_OVERLAP;
  return MFSDP_OK;
}

}  // namespace

int check_step_args(const mfsdp_matrix_shard* shards, int32_t n_shards, const void* grad, int32_t grad_dtype,
                    const float* momentum, const void* update, int32_t update_dtype, int64_t numel, double beta,
                    int32_t nesterov, int32_t ns_steps, double a, double b, double c, double eps,
                    size_t* workspace_bytes) {
  Layout L;
  const int st = validate_step_args(shards, n_shards, grad, grad_dtype, momentum, update, update_dtype, numel, beta,
                                    nesterov, ns_steps, a, b, c, eps, &L);
  if (workspace_bytes) *workspace_bytes = (st == MFSDP_OK && n_shards > 0) ? L.bytes : 0;
  return st;
}

}  // namespace mfsdp

extern "C" int mfsdp_muon_owner_step_phases(const mfsdp_matrix_shard* shards, int32_t n_shards,
                                            const void* grad, int32_t grad_dtype, float* momentum, void* update,
                                            int32_t update_dtype, int64_t numel, double beta_d, int32_t nesterov,
                                            int32_t ns_steps, double a_d, double b_d, double c_d, double eps_d,
                                            void* workspace, size_t workspace_bytes, void* stream_ptr,
                                            int32_t phases) {
  if (phases <= 0 || (phases & ~(MFSDP_PHASE_MOMENTUM | MFSDP_PHASE_NEWTON_SCHULZ)) != 0)
    return MFSDP_ERR_INVALID_ARG;
  Layout L;
  int st = validate_step(shards, n_shards, grad, grad_dtype, momentum, update, update_dtype, numel, beta_d, nesterov,
                         ns_steps, a_d, b_d, c_d, eps_d, workspace, workspace_bytes, &L);
  if (st != MFSDP_OK || n_shards == 0) return st;
  const float beta = (float)beta_d, a = (float)a_d, b = (float)b_d, c = (float)c_d, eps = (float)eps_d;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (phases & MFSDP_PHASE_MOMENTUM) {
    st = clear_status(ws, stream);
    if (st != MFSDP_OK) return st;
    st = launch_momentum_phase(shards, n_shards, L, grad, grad_dtype, momentum, beta, nesterov, eps, ws, stream);
    if (st != MFSDP_OK) return st;
  }
  if (phases & MFSDP_PHASE_NEWTON_SCHULZ) {
    st = launch_ns_phase(shards, n_shards, L, update, update_dtype, ns_steps, a, b, c, ws, stream);
    if (st != MFSDP_OK) return st;
  }
  return MFSDP_OK;
}

extern "C" int mfsdp_muon_owner_step_apply(const mfsdp_matrix_shard* shards, int32_t n_shards, const void* grad,
                                           int32_t grad_dtype, float* momentum, void* update, int32_t update_dtype,
                                           void* weights, int32_t weight_dtype, int64_t numel, double beta,
                                           int32_t nesterov, int32_t ns_steps, double a, double b, double c,
                                           double eps, double lr, double weight_decay, int32_t scale_mode,
                                           void* workspace, size_t workspace_bytes, void* stream_ptr) {
  if (weight_dtype != MFSDP_DTYPE_F32 && weight_dtype != MFSDP_DTYPE_BF16) return MFSDP_ERR_UNSUPPORTED_DTYPE;
  if (scale_mode < 0 || scale_mode > 2 || !std::isfinite(lr) || !std::isfinite(weight_decay) || ns_steps < 1)
    return MFSDP_ERR_INVALID_ARG;
  // The weights stand in for the update buffer in the common checks when no
  // update is requested; both are checked against each other below.
  void* checked = update ? update : weights;
  const int32_t checked_dtype = update ? update_dtype : weight_dtype;
  Layout L;
  int st = validate_step(shards, n_shards, grad, grad_dtype, momentum, checked, checked_dtype, numel, beta, nesterov,
                         ns_steps, a, b, c, eps, workspace, workspace_bytes, &L);
  if (st != MFSDP_OK || n_shards == 0) return st;
  if (!weights) return MFSDP_ERR_INVALID_ARG;
  if (!aligned(weights, 16)) return MFSDP_ERR_MISALIGNED;
  const size_t wbytes = (size_t)numel * dtype_size(weight_dtype);
  if (ranges_overlap(weights, wbytes, grad, (size_t)numel * dtype_size(grad_dtype)) ||
      ranges_overlap(weights, wbytes, momentum, (size_t)numel * 4) ||
      ranges_overlap(weights, wbytes, workspace, L.bytes) ||
      (update && ranges_overlap(weights, wbytes, update, (size_t)numel * dtype_size(update_dtype))))
    return MFSDP_ERR_OVERLAP;
  const float fb = (float)beta, fe = (float)eps;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  st = clear_status(ws, stream);
  if (st != MFSDP_OK) return st;
  st = launch_momentum_phase(shards, n_shards, L, grad, grad_dtype, momentum, fb, nesterov, fe, ws, stream);
  if (st != MFSDP_OK) return st;
  ApplyArgs ap{weights, weight_dtype, lr, weight_decay, scale_mode};
  return launch_ns_phase(shards, n_shards, L, update, update_dtype, ns_steps, (float)a, (float)b, (float)c, ws, stream,
                         &ap);
}

namespace {

// Balanced groups over the shards marked in `member`: offset order, cut where
// the running Newton-Schulz cost crosses k/ng of their total, so each group
// is one contiguous range of the flat buffers (apart from shards placed in
// other groups) and the groups' compute is balanced.  Group ids start at
// `first`; returns the number of non-empty groups.
int balanced_groups(const mfsdp_matrix_shard* shards, int n, const std::vector<char>& member, int ng, int first,
                    std::vector<int>& group_of) {
  std::vector<int> ord;
  for (int i = 0; i < n; ++i)
    if (member[i]) ord.push_back(i);
  if (ord.empty()) return 0;
  std::sort(ord.begin(), ord.end(), [&](int x, int y) { return shards[x].offset < shards[y].offset; });
  std::vector<double> cost(ord.size());
  double total = 0.0;
  for (size_t k = 0; k < ord.size(); ++k) {
    const mfsdp_matrix_shard& sh = shards[ord[k]];
    const double sm = (double)std::min(sh.rows, sh.cols), l = (double)std::max(sh.rows, sh.cols);
    cost[k] = 4.0 * sm * sm * l + 2.0 * sm * sm * sm + sm * l;   // + s*l: the momentum pass
    total += cost[k];
  }
  ng = std::min<int>(ng, (int)ord.size());
  std::vector<int> slot(ord.size()), used(ng, 0);
  double run = 0.0;
  for (size_t k = 0; k < ord.size(); ++k) {
    int g = total > 0.0 ? (int)(run / total * ng) : 0;
    g = std::min(std::max(g, 0), ng - 1);
    slot[k] = g;
    used[g] = 1;
    run += cost[k];
  }
  std::vector<int> remap(ng);
  int nz = 0;
  for (int g = 0; g < ng; ++g) remap[g] = used[g] ? nz++ : -1;
  for (size_t k = 0; k < ord.size(); ++k) group_of[ord[k]] = first + remap[slot[k]];
  return nz;
}

// Shard groups of the host-buffer step, in execution order; group_of[i] is
// shard i's group.  groups >= 1: balanced groups over all shards.
// groups == 0: the copy volume decides (mfsdp_host_step_groups).  Only the
// first copy in and the last copy out are exposed; every group past the first
// costs a little compute.
//  - Large sets (g >= 6): g balanced groups, each of which still fills the
//    GPU, between a small head and a small tail group: up to two of the
//    smallest shards with the largest short side (the most Newton-Schulz work
//    per byte) at each end, at most 1/(2g) of the elements each.  The head's
//    compute hides the next group's copy in, the tail's the copy out before it.
//  - Mid-sized sets (3 <= g <= 5): a ramp -- shards ordered small -> large ->
//    small by size and cut at 4 %, 28 %, 72 % and 96 % of the bytes -- which
//    makes the two exposed copies small with five groups, where balanced
//    groups of a few matrices would leave most of the GPU idle.
int plan_host_groups(const mfsdp_matrix_shard* shards, int n, int groups, size_t elem_bytes,
                     std::vector<int>& group_of) {
  group_of.assign(n, 0);
  if (n <= 0) return 1;
  std::vector<char> all(n, 1);
  if (groups >= 1) return balanced_groups(shards, n, all, groups, 0, group_of);
  double elems = 0.0;
  for (int i = 0; i < n; ++i) elems += (double)shards[i].rows * (double)shards[i].cols;
  const long g = std::lround(std::sqrt(elems * (double)elem_bytes / 50e6));
  if (g <= 1) return 1;
  if (g == 2 || n < 5) return balanced_groups(shards, n, all, (int)g, 0, group_of);
  if (g >= 6) {
    const int gm = (int)std::min<long>(g, 16);
    int64_t smax = 0;
    for (int i = 0; i < n; ++i) smax = std::max(smax, std::min(shards[i].rows, shards[i].cols));
    std::vector<int> cand;
    for (int i = 0; i < n; ++i)
      if (std::min(shards[i].rows, shards[i].cols) == smax) cand.push_back(i);
    std::sort(cand.begin(), cand.end(), [&](int x, int y) {
      const int64_t nx = shards[x].rows * shards[x].cols, ny = shards[y].rows * shards[y].cols;
      return nx != ny ? nx < ny : shards[x].offset < shards[y].offset;
    });
    const double limit = elems / (2.0 * gm);
    std::vector<int> head, tail;
    size_t k = 0;
    for (std::vector<int>* end : {&head, &tail}) {
      double e = 0.0;
      while (k < cand.size() && end->size() < 2) {
        const double ne = (double)shards[cand[k]].rows * (double)shards[cand[k]].cols;
        if (e + ne > limit) break;
        end->push_back(cand[k++]);
        e += ne;
      }
    }
    if (head.empty() || tail.empty()) return balanced_groups(shards, n, all, gm, 0, group_of);
    std::vector<char> mid(n, 1);
    for (int i : head) { mid[i] = 0; group_of[i] = 0; }
    for (int i : tail) mid[i] = 0;
    const int nm = balanced_groups(shards, n, mid, gm, 1, group_of);
    for (int i : tail) group_of[i] = 1 + nm;
    return 2 + nm;
  }
  std::vector<int> by(n);
  for (int i = 0; i < n; ++i) by[i] = i;
  std::sort(by.begin(), by.end(), [&](int x, int y) {
    const int64_t nx = shards[x].rows * shards[x].cols, ny = shards[y].rows * shards[y].cols;
    return nx != ny ? nx < ny : shards[x].offset < shards[y].offset;
  });
  // small -> large: the even positions; large -> small: the odd ones reversed
  std::vector<int> seq;
  for (int k = 0; k < n; k += 2) seq.push_back(by[k]);
  for (int k = (n % 2 == 0) ? n - 1 : n - 2; k >= 1; k -= 2) seq.push_back(by[k]);
  const double cuts[4] = {0.04, 0.28, 0.72, 0.96};
  std::vector<int> slot(n);
  bool used[5] = {false, false, false, false, false};
  double run = 0.0;
  for (int i : seq) {
    const double e = (double)shards[i].rows * (double)shards[i].cols;
    const double mid = (run + 0.5 * e) / elems;          // a shard goes where its midpoint falls
    int k = 0;
    while (k < 4 && cuts[k] <= mid) ++k;
    slot[i] = k;
    used[k] = true;
    run += e;
  }
  int remap[5], ng = 0;                                    // a large shard can leave a slot empty
  for (int k = 0; k < 5; ++k) remap[k] = used[k] ? ng++ : -1;
  for (int i = 0; i < n; ++i) group_of[i] = remap[slot[i]];
  return ng;
}

}  // namespace

extern "C" int32_t mfsdp_host_step_groups(const mfsdp_matrix_shard* shards, int32_t n_shards, int32_t grad_dtype,
                                          int32_t update_dtype, int32_t groups, int32_t* group_of) {
  const auto known = [](int32_t dt) { return dt == MFSDP_DTYPE_F32 || dt == MFSDP_DTYPE_BF16; };
  if (!shards || n_shards <= 0 || groups < 0 || !known(grad_dtype) || !known(update_dtype)) return 0;
  std::vector<int> gof;
  const int ng = plan_host_groups(shards, n_shards, groups, dtype_size(grad_dtype) + dtype_size(update_dtype), gof);
  if (group_of)
    for (int i = 0; i < n_shards; ++i) group_of[i] = gof[i];
  return ng;
}

extern "C" int mfsdp_muon_owner_step_host(const mfsdp_matrix_shard* shards, int32_t n_shards, const void* grad_host,
                                          void* grad_dev, int32_t grad_dtype, float* momentum, void* update_dev,
                                          void* update_host, int32_t update_dtype, int64_t numel, double beta_d,
                                          int32_t nesterov, int32_t ns_steps, double a_d, double b_d, double c_d,
                                          double eps_d, void* workspace, size_t workspace_bytes, int32_t groups,
                                          void* stream_ptr) {
  if (groups < 0) return MFSDP_ERR_INVALID_ARG;
  Layout L;
  int st = validate_step(shards, n_shards, grad_dev, grad_dtype, momentum, update_dev, update_dtype, numel, beta_d,
                         nesterov, ns_steps, a_d, b_d, c_d, eps_d, workspace, workspace_bytes, &L);
  if (st != MFSDP_OK || n_shards == 0) return st;
  if (!grad_host || !update_host) return MFSDP_ERR_INVALID_ARG;
  const float beta = (float)beta_d, a = (float)a_d, b = (float)b_d, c = (float)c_d, eps = (float)eps_d;
  const size_t gsz = dtype_size(grad_dtype), usz = dtype_size(update_dtype);

  // Groups (in execution order) and, per group, the element ranges to copy:
  // runs of its shards that are neighbours in offset order, so a group whose
  // shards are contiguous in the flat buffers costs one copy each way.
  std::vector<int> gof;
  const int ng = plan_host_groups(shards, n_shards, groups, gsz + usz, gof);
  std::vector<std::vector<mfsdp_matrix_shard>> grp(ng);
  std::vector<std::vector<std::pair<int64_t, int64_t>>> runs(ng);
  std::vector<int> ord(n_shards);
  for (int i = 0; i < n_shards; ++i) ord[i] = i;
  std::sort(ord.begin(), ord.end(), [&](int x, int y) { return shards[x].offset < shards[y].offset; });
  for (int k = 0; k < n_shards; ++k) {
    const int i = ord[k], g = gof[i];
    const int64_t lo = shards[i].offset, hi = lo + shards[i].rows * shards[i].cols;
    grp[g].push_back(shards[i]);
    if (k > 0 && gof[ord[k - 1]] == g) runs[g].back().second = std::max(runs[g].back().second, hi);
    else runs[g].push_back({lo, hi});
  }

  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxPipeDevices) return MFSDP_ERR_CUDA;
  // The device's copy streams and events, kept for the life of the process
  // (creating streams per call occasionally stalled a call for hundreds of
  // ms).  Calls on one device enqueue under its lock and share the copy
  // streams, so their copies run in call order.
  CopyPipe& pipe = g_pipe[dev];
  std::lock_guard<std::mutex> lock(pipe.mu);
  if (!pipe.s_in && (cudaStreamCreateWithFlags(&pipe.s_in, cudaStreamNonBlocking) != cudaSuccess ||
                     cudaStreamCreateWithFlags(&pipe.s_out, cudaStreamNonBlocking) != cudaSuccess))
    return MFSDP_ERR_CUDA;
  // ev[0]: entry; per group: copied in, computed, copied out.  Re-recording an
  // event that earlier calls' enqueued waits refer to is fine: those waits
  // hold the state the event had when they were enqueued.
  std::vector<cudaEvent_t>& ev = pipe.ev;
  while (ev.size() < 1 + 3 * (size_t)ng) {
    cudaEvent_t e = nullptr;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return MFSDP_ERR_CUDA;
    ev.push_back(e);
  }
  cudaStream_t s_in = pipe.s_in, s_out = pipe.s_out;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (clear_status(ws, stream) != MFSDP_OK) return MFSDP_ERR_CUDA;
  cudaError_t ce = cudaEventRecord(ev[0], stream);            // earlier work on `stream` comes first
  ce = ce == cudaSuccess ? cudaStreamWaitEvent(s_in, ev[0], 0) : ce;
  for (int g = 0; g < ng && ce == cudaSuccess && st == MFSDP_OK; ++g) {
    const std::vector<mfsdp_matrix_shard>& sh = grp[g];
    if (sh.empty()) continue;
    const PhaseRange range("mfsdp host-buffer group");
    cudaEvent_t e_in = ev[1 + 3 * g], e_done = ev[2 + 3 * g], e_out = ev[3 + 3 * g];
    for (size_t r = 0; r < runs[g].size() && ce == cudaSuccess; ++r) {
      const int64_t lo = runs[g][r].first, hi = runs[g][r].second;
      ce = cudaMemcpyAsync(static_cast<uint8_t*>(grad_dev) + (size_t)lo * gsz,
                           static_cast<const uint8_t*>(grad_host) + (size_t)lo * gsz, (size_t)(hi - lo) * gsz,
                           cudaMemcpyHostToDevice, s_in);
    }
    if (ce == cudaSuccess) ce = cudaEventRecord(e_in, s_in);
    if (ce == cudaSuccess) ce = cudaStreamWaitEvent(stream, e_in, 0);
    if (ce != cudaSuccess) break;
    Layout Lg;
    st = make_layout(sh.data(), (int)sh.size(), &Lg);        // fits: never larger than the whole set's layout
    if (st != MFSDP_OK) break;
    st = launch_momentum_phase(sh.data(), (int)sh.size(), Lg, grad_dev, grad_dtype, momentum, beta, nesterov, eps, ws,
                               stream);
    if (st != MFSDP_OK) break;
    st = launch_ns_phase(sh.data(), (int)sh.size(), Lg, update_dev, update_dtype, ns_steps, a, b, c, ws, stream);
    if (st != MFSDP_OK) break;
    ce = cudaEventRecord(e_done, stream);
    if (ce == cudaSuccess) ce = cudaStreamWaitEvent(s_out, e_done, 0);
    for (size_t r = 0; r < runs[g].size() && ce == cudaSuccess; ++r) {
      const int64_t lo = runs[g][r].first, hi = runs[g][r].second;
      ce = cudaMemcpyAsync(static_cast<uint8_t*>(update_host) + (size_t)lo * usz,
                           static_cast<const uint8_t*>(update_dev) + (size_t)lo * usz, (size_t)(hi - lo) * usz,
                           cudaMemcpyDeviceToHost, s_out);
    }
    if (ce == cudaSuccess) ce = cudaEventRecord(e_out, s_out);
  }
  // `stream` ends after every copy out.  The waits come after the loop: inside
  // it they would hold group g+1's compute until group g's update has left the
  // device, serialising every copy out with the next group's compute (the
  // ranges they touch are disjoint: a group's copy out reads only its own
  // update segments).
  for (int g = 0; g < ng && ce == cudaSuccess; ++g)
    if (!grp[g].empty()) ce = cudaStreamWaitEvent(stream, ev[3 + 3 * g], 0);
  if (ce != cudaSuccess) return MFSDP_ERR_CUDA;
  return st;
}

extern "C" int mfsdp_muon_owner_step(const mfsdp_matrix_shard* shards, int32_t n_shards, const void* grad,
                                     int32_t grad_dtype, float* momentum, void* update, int32_t update_dtype,
                                     int64_t numel, double beta, int32_t nesterov, int32_t ns_steps, double a,
                                     double b, double c, double eps, void* workspace, size_t workspace_bytes,
                                     void* stream) {
  return mfsdp_muon_owner_step_phases(shards, n_shards, grad, grad_dtype, momentum, update, update_dtype, numel,
                                      beta, nesterov, ns_steps, a, b, c, eps, workspace, workspace_bytes, stream,
                                      MFSDP_PHASE_MOMENTUM | MFSDP_PHASE_NEWTON_SCHULZ);
}

namespace mfsdp {
namespace {

int launch_momentum_phase(const mfsdp_matrix_shard* shards, int n_shards, const Layout& L, const void* grad,
                          int32_t grad_dtype, float* momentum, float beta, int32_t nesterov, float eps, uint8_t* ws,
                          cudaStream_t stream) {
  const PhaseRange range("mfsdp momentum");
  float2* norm = reinterpret_cast<float2*>(ws + L.norm_off);
  float* partials = reinterpret_cast<float*>(ws + L.partial_off);
  const size_t gsz = dtype_size(grad_dtype);
  int st = MFSDP_OK;
  for (int base = 0; base < n_shards; base += kMaxBatch) {
    const int cnt = std::min(kMaxBatch, n_shards - base);
    MomBatch mb;
    std::memset(&mb, 0, sizeof(mb));
    mb.n = cnt;
    mb.grad_bf16 = grad_dtype == MFSDP_DTYPE_BF16;
    mb.nesterov = nesterov;
    mb.beta = beta;
    mb.partials = partials;
    int tiles = 0;
    for (int k = 0; k < cnt; ++k) {
      const int i = base + k;
      const mfsdp_matrix_shard& sh = shards[i];
      const MatLayout& m = L.mats[i];
      MomMat& d = mb.mat[k];
      d.g = static_cast<const uint8_t*>(grad) + (size_t)sh.offset * gsz;
      d.m = momentum + sh.offset;
      d.y = ws + m.x0;
      d.rows = sh.rows;
      d.cols = sh.cols;
      d.s_pad = m.s_pad;
      d.l_pad = m.l_pad;
      d.transposed = m.transposed;
      d.vec_ok = (sh.offset % 8 == 0) && (sh.cols % 8 == 0);
      d.g32 = aligned(d.g, 32);
      d.m32 = aligned(d.m, 32);
      d.tiles_j = m.l_pad / kTile;
      d.partial0 = m.partial0;
      mb.tile_start[k] = tiles;
      tiles += m.tiles_k1;
    }
    mb.tile_start[cnt] = tiles;
    st = cuda_status(launch_momentum(mb, tiles, stream));
    if (st != MFSDP_OK) return st;
  }
  for (int base = 0; base < n_shards; base += kMaxBatch) {
    const int cnt = std::min(kMaxBatch, n_shards - base);
    NormBatch nb;
    std::memset(&nb, 0, sizeof(nb));
    nb.n = cnt;
    nb.first = base;
    nb.eps = eps;
    nb.partials = partials;
    nb.norm = norm;
    for (int k = 0; k < cnt; ++k) nb.start[k] = L.mats[base + k].partial0 * kPartialsPerTile;
    nb.start[cnt] = (L.mats[base + cnt - 1].partial0 + L.mats[base + cnt - 1].tiles_k1) * kPartialsPerTile;
    st = cuda_status(launch_norm_finalize(nb, stream));
    if (st != MFSDP_OK) return st;
  }
  return MFSDP_OK;
}

int launch_ns_phase(const mfsdp_matrix_shard* shards, int n_shards, const Layout& L, void* update,
                    int32_t update_dtype, int32_t ns_steps, float a, float b, float c, uint8_t* ws,
                    cudaStream_t stream, const ApplyArgs* apply) {
  const PhaseRange range(ns_steps ? "mfsdp newton-schulz" : "mfsdp emit");
  float2* norm = reinterpret_cast<float2*>(ws + L.norm_off);
  int32_t* status = reinterpret_cast<int32_t*>(ws);
  const size_t usz = dtype_size(update_dtype);
  int st = MFSDP_OK;
  if (ns_steps == 0) {
    for (int base = 0; base < n_shards; base += kMaxBatch) {
      const int cnt = std::min(kMaxBatch, n_shards - base);
      EmitBatch eb;
      std::memset(&eb, 0, sizeof(eb));
      eb.n = cnt;
      eb.out_bf16 = update_dtype == MFSDP_DTYPE_BF16;
      eb.norm = norm;
      int tiles = 0;
      for (int k = 0; k < cnt; ++k) {
        const int i = base + k;
        const MatLayout& m = L.mats[i];
        EmitMat& d = eb.mat[k];
        d.y = ws + m.x0;
        d.out = static_cast<uint8_t*>(update) + (size_t)shards[i].offset * usz;
        d.rows = shards[i].rows;
        d.cols = shards[i].cols;
        d.s_pad = m.s_pad;
        d.tiles_j = m.l_pad / kTile;
        d.transposed = m.transposed;
        d.norm_idx = i;
        eb.tile_start[k] = tiles;
        tiles += m.tiles_k1;
      }
      eb.tile_start[cnt] = tiles;
      st = cuda_status(launch_emit(eb, tiles, stream));
      if (st != MFSDP_OK) return st;
    }
    return MFSDP_OK;
  }

  // ------------------------------------------------------- Newton-Schulz
  // One persistent launch per batch runs all 3 * ns_steps products; its tile
  // counter and completion counters start at zero.
  int32_t* counters = reinterpret_cast<int32_t*>(ws + L.done_off);
  for (int base = 0; base < n_shards; base += kMaxBatch) {
    const int cnt = std::min(kMaxBatch, n_shards - base);
    NsBatch nb;
    std::memset(&nb, 0, sizeof(nb));
    nb.n = cnt;
    nb.ns_steps = ns_steps;
    nb.phase_begin = 0;
    nb.phase_end = 3 * ns_steps;   // + 1 below when a Gram-space matrix has its final product
    nb.out_bf16 = update_dtype == MFSDP_DTYPE_BF16;
    nb.a = a;
    nb.b = b;
    nb.c = c;
    nb.norm = norm;
    nb.ws = ws;
    nb.status = status;
    nb.wait_limit_ns = 0;   // set by launch_ns from the launch's products and the device's CTA pairs
    nb.next_tile = counters;
    nb.done = counters + 1 + base;
    if (apply) {
      nb.decay = (float)(1.0 - apply->lr * apply->wd);
      nb.w_bf16 = apply->w_dtype == MFSDP_DTYPE_BF16;
    }
    nb.narrow = use_narrow_tiles(L, base, cnt, &nb.narrow_mask) ? 1 : 0;
    const int width_sym = (nb.narrow_mask >> kGram) & 1 ? kBlockN / 2 : kBlockN;
    const int width_upd = (nb.narrow_mask >> kUpdate) & 1 ? kBlockN / 2 : kBlockN;
    for (int k = 0; k < cnt; ++k) {
      const int i = base + k;
      const MatLayout& m = L.mats[i];
      NsMat& d = nb.mat[k];
      d.x[0] = ws + m.x0;
      d.x[1] = ws + m.x1;
      d.a = ws + m.a;
      d.b = ws + m.b;
      d.gram_space = use_gram_space(m, ns_steps) ? 1 : 0;
      d.c = ws + m.c;
      d.q[0] = ws + m.q0;
      d.q[1] = ws + m.q1;
      if (d.gram_space) nb.phase_end = 3 * ns_steps + 1;
      d.out = update ? static_cast<void*>(static_cast<uint8_t*>(update) + (size_t)shards[i].offset * usz) : nullptr;
      if (apply) {
        d.w = static_cast<uint8_t*>(apply->w) + (size_t)shards[i].offset * dtype_size(apply->w_dtype);
        d.lr_scale = (float)(apply->lr * shape_scale(shards[i].rows, shards[i].cols, apply->scale_mode));
      }
      d.s_pad = m.s_pad;
      d.l_pad = m.l_pad;
      d.s = m.s;
      d.l = m.l;
      const GemmTiling ts = gemm_tiling(kGram, m.s_pad, m.l_pad, width_sym);
      const GemmTiling tu = gemm_tiling(kUpdate, m.s_pad, m.l_pad, width_upd);
      d.tiles_sym = ts.tiles;
      d.tiles_m = tu.tiles_m;
      d.tiles_n = tu.tiles_n;
      d.n_last = tu.n_last;
      d.norm_idx = i;
      d.transposed = m.transposed;
      d.vec_ok = (shards[i].offset % 8 == 0) && ((m.transposed ? m.s : m.l) % 8 == 0);
    }
    // Inside each product, longest K first: the persistent pairs take tiles
    // round-robin, so the last rounds hold the cheapest tiles.  Products 0-2
    // repeat every iteration; product 3, after the last iteration, holds the
    // Gram-space matrices' final X = Q X0.
    int32_t off = 0;
    for (int prod = 0; prod <= 3; ++prod) {
      std::vector<int> order(cnt);
      for (int k = 0; k < cnt; ++k) order[k] = k;
      auto kb_of = [&](int k) {
        const NsMat& d = nb.mat[k];
        return prod == kGram && !d.gram_space ? d.l_pad : d.s_pad;
      };
      auto tiles_of = [&](const NsMat& d) {
        if (prod == 3) return d.gram_space ? d.tiles_m * d.tiles_n : 0;
        if (prod == 2) return d.gram_space ? 2 * d.tiles_sym : d.tiles_m * d.tiles_n;
        return d.tiles_sym;
      };
      std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return kb_of(x) > kb_of(y); });
      if (prod < 3) nb.mode_start[prod] = off;
      int32_t tiles = 0;
      for (int j = 0; j < cnt; ++j) {
        const NsMat& d = nb.mat[order[j]];
        nb.order[prod][j] = (uint8_t)order[j];
        nb.tile_start[prod][j] = tiles;
        tiles += tiles_of(d);
      }
      nb.tile_start[prod][cnt] = tiles;
      if (prod < 3) off += tiles;
      else nb.tile_end = off * ns_steps + tiles;
    }
    nb.iter_tiles = off;
    nb.final_start = off * ns_steps;
    nb.tile_begin = 0;
    nb.stall_tile = g_stall_tile.exchange(-1);
    st = cuda_status(cudaMemsetAsync(counters, 0, sizeof(int32_t) * (size_t)(n_shards + 1), stream));
    if (st != MFSDP_OK) return st;
    st = cuda_status(launch_ns(nb, L.bytes, stream));
    if (st != MFSDP_OK) return st;
  }
  return MFSDP_OK;
}

}  // namespace
}  // namespace mfsdp

extern "C" int mfsdp_muon_step_flops(const mfsdp_matrix_shard* shards, int32_t n_shards, int32_t ns_steps,
                                     uint64_t* dense, uint64_t* executed) {
  if (ns_steps < 0 || ns_steps > 64 || !dense || !executed) return MFSDP_ERR_INVALID_ARG;
  Layout L;
  const int st = make_layout(shards, n_shards, &L);
  if (st != MFSDP_OK) return st;
  uint64_t dn = 0, ex = 0;
  for (int i = 0; i < n_shards; ++i) {
    const MatLayout& m = L.mats[i];
    const uint64_t s = (uint64_t)m.s, l = (uint64_t)m.l;
    dn += (uint64_t)ns_steps * (4 * s * s * l + 2 * s * s * s);
    const uint64_t gram = executed_flops(kGram, m.s, m.s_pad, m.l_pad), sym = executed_flops(kPoly, m.s, m.s_pad, m.l_pad),
                   upd = executed_flops(kUpdate, m.s, m.s_pad, m.l_pad);
    if (use_gram_space(m, ns_steps))   // A_0, T P_k, T-1 each of C, A and Q, the final Q X0
      ex += gram + (uint64_t)ns_steps * sym + 3ull * (uint64_t)(ns_steps - 1) * sym + upd;
    else
      ex += (uint64_t)ns_steps * (gram + sym + upd);
  }
  *dense = dn;
  *executed = ex;
  return MFSDP_OK;
}

extern "C" int mfsdp_muon_gram_space_layout(const mfsdp_matrix_shard* shards, int32_t n_shards, int32_t ns_steps,
                                            int64_t* out) {
  if (ns_steps < 0 || ns_steps > 64) return MFSDP_ERR_INVALID_ARG;
  Layout L;
  const int st = make_layout(shards, n_shards, &L);
  if (st != MFSDP_OK) return st;
  if (n_shards > 0 && !out) return MFSDP_ERR_INVALID_ARG;
  for (int i = 0; i < n_shards; ++i) {
    const MatLayout& m = L.mats[i];
    int64_t* o = out + 4 * i;
    o[0] = use_gram_space(m, ns_steps) ? 1 : 0;
    o[1] = (int64_t)m.c; o[2] = (int64_t)m.q0; o[3] = (int64_t)m.q1;
  }
  return MFSDP_OK;
}

extern "C" int mfsdp_test_inject_stall(int32_t tile) {
  if (tile < 0) return MFSDP_ERR_INVALID_ARG;
  g_stall_tile.store(tile);
  return MFSDP_OK;
}

extern "C" int mfsdp_muon_device_status(const void* workspace, void* stream_ptr, int32_t* detail) {
  if (!workspace) return MFSDP_ERR_INVALID_ARG;
  int32_t word = 0;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return MFSDP_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MFSDP_ERR_CUDA;
  if (detail) *detail = word;
  return word ? MFSDP_ERR_DEVICE_TIMEOUT : MFSDP_OK;
}

extern "C" int mfsdp_adamw_tail_step(float* p, const float* g, float* m, float* v, int64_t n, double lr,
                                     double beta1, double beta2, double eps, double wd, int64_t step,
                                     void* stream_ptr) {
  if (n < 0 || step < 1) return MFSDP_ERR_INVALID_ARG;
  if (!(beta1 >= 0.0 && beta1 < 1.0) || !(beta2 >= 0.0 && beta2 < 1.0)) return MFSDP_ERR_INVALID_ARG;
  if (!std::isfinite(lr) || !std::isfinite(eps) || !std::isfinite(wd)) return MFSDP_ERR_INVALID_ARG;
  if (n == 0) return MFSDP_OK;
  if (!p || !g || !m || !v) return MFSDP_ERR_INVALID_ARG;
  if (!aligned(p, 16) || !aligned(g, 16) || !aligned(m, 16) || !aligned(v, 16)) return MFSDP_ERR_MISALIGNED;
  const size_t nb = (size_t)n * 4;
  const void* bufs[4] = {p, g, m, v};
  for (int i = 0; i < 4; ++i)
    for (int j = i + 1; j < 4; ++j)
      if (ranges_overlap(bufs[i], nb, bufs[j], nb)) return MFSDP_ERR_OVERLAP;
  const double bc1 = 1.0 - std::pow(beta1, (double)step);
  const double bc2 = 1.0 - std::pow(beta2, (double)step);
  AdamScalars k;
  k.decay = (float)(1.0 - lr * wd);
  k.beta1 = (float)beta1;
  k.beta2 = (float)beta2;
  k.omb1 = (float)(1.0 - beta1);
  k.omb2 = (float)(1.0 - beta2);
  k.step_size = (float)(lr / bc1);
  k.inv_sqrt_bc2 = (float)(1.0 / std::sqrt(bc2));
  k.eps = (float)eps;
  const PhaseRange range("mfsdp adamw tail");
  return cuda_status(launch_adamw(p, g, m, v, n, k, static_cast<cudaStream_t>(stream_ptr)));
}

// ------------------------------------------------------------------ owner segments
extern "C" int mfsdp_model_layout(const mfsdp_param* params, int32_t n_params, int64_t align_elems, int64_t* offsets,
                                  int64_t* total) {
  if (n_params < 0 || align_elems < 1 || !total || (n_params > 0 && (!params || !offsets)))
    return MFSDP_ERR_INVALID_ARG;
  int64_t off = 0;
  for (int i = 0; i < n_params; ++i) {
    if (params[i].rows < 1 || params[i].cols < 1 || params[i].rows > INT64_MAX / params[i].cols)
      return MFSDP_ERR_UNSUPPORTED_SHAPE;
    off = (off + align_elems - 1) / align_elems * align_elems;
    offsets[i] = off;
    off += params[i].rows * params[i].cols;
  }
  *total = (off + align_elems - 1) / align_elems * align_elems;
  return MFSDP_OK;
}

extern "C" int mfsdp_placement_segments(const mfsdp_placement* src, int32_t n_src, const mfsdp_placement* dst,
                                        int32_t n_dst, int32_t dst_owner, mfsdp_segment* out, int32_t* n_out) {
  if (n_src < 0 || n_dst < 0 || !n_out || (n_src > 0 && !src) || (n_dst > 0 && (!dst || !out)))
    return MFSDP_ERR_INVALID_ARG;
  std::vector<int> by_param;
  for (int i = 0; i < n_src; ++i) {
    const int pid = src[i].param_id;
    if (pid < 0 || src[i].numel < 0 || src[i].offset < 0) return MFSDP_ERR_INVALID_ARG;
    if ((int)by_param.size() <= pid) by_param.resize(pid + 1, -1);
    if (by_param[pid] >= 0) return MFSDP_ERR_INVALID_ARG;   // a parameter placed twice
    by_param[pid] = i;
  }
  std::vector<int> mine;
  for (int i = 0; i < n_dst; ++i)
    if (dst[i].owner == dst_owner) mine.push_back(i);
  std::sort(mine.begin(), mine.end(), [&](int x, int y) { return dst[x].offset < dst[y].offset; });
  int k = 0;
  for (int i : mine) {
    const int pid = dst[i].param_id;
    if (pid < 0 || pid >= (int)by_param.size() || by_param[pid] < 0) return MFSDP_ERR_INVALID_ARG;
    const mfsdp_placement& f = src[by_param[pid]];
    if (f.numel != dst[i].numel) return MFSDP_ERR_INVALID_ARG;
    mfsdp_segment& g = out[k++];
    std::memset(&g, 0, sizeof(g));
    g.src_offset = f.offset;
    g.dst_offset = dst[i].offset;
    g.numel = f.numel;
    g.src_index = f.owner;
  }
  *n_out = k;
  return MFSDP_OK;
}

extern "C" int mfsdp_segment_copy(const void* const* srcs, const int64_t* src_numel, int32_t n_src, int32_t src_dtype,
                                  const mfsdp_segment* segs, int32_t n_segs, int32_t mode, void* dst,
                                  int32_t dst_dtype, int64_t dst_numel, void* stream_ptr) {
  if (n_src < 1 || n_src > kMaxSources || !srcs || !src_numel || n_segs < 0 || (n_segs > 0 && !segs) ||
      (mode != MFSDP_SEGMENT_REDUCE && mode != MFSDP_SEGMENT_GATHER) || dst_numel < 0)
    return MFSDP_ERR_INVALID_ARG;
  if ((src_dtype != MFSDP_DTYPE_F32 && src_dtype != MFSDP_DTYPE_BF16) ||
      (dst_dtype != MFSDP_DTYPE_F32 && dst_dtype != MFSDP_DTYPE_BF16))
    return MFSDP_ERR_UNSUPPORTED_DTYPE;
  if (n_segs == 0) return MFSDP_OK;
  if (!dst) return MFSDP_ERR_INVALID_ARG;
  if (!aligned(dst, 16)) return MFSDP_ERR_MISALIGNED;
  for (int k = 0; k < n_src; ++k) {
    if (!srcs[k] || src_numel[k] < 0) return MFSDP_ERR_INVALID_ARG;
    if (!aligned(srcs[k], 16)) return MFSDP_ERR_MISALIGNED;
    if (ranges_overlap(dst, (size_t)dst_numel * dtype_size(dst_dtype), srcs[k],
                       (size_t)src_numel[k] * dtype_size(src_dtype)))
      return MFSDP_ERR_OVERLAP;
  }
  int64_t min_src = INT64_MAX;
  for (int k = 0; k < n_src; ++k) min_src = std::min(min_src, src_numel[k]);
  for (int i = 0; i < n_segs; ++i) {
    const mfsdp_segment& g = segs[i];
    if (g.numel < 0 || g.src_offset < 0 || g.dst_offset < 0) return MFSDP_ERR_INVALID_ARG;
    if (mode == MFSDP_SEGMENT_GATHER && (g.src_index < 0 || g.src_index >= n_src)) return MFSDP_ERR_INVALID_ARG;
    const int64_t lim = mode == MFSDP_SEGMENT_GATHER ? src_numel[g.src_index] : min_src;
    if (g.src_offset > lim || g.numel > lim - g.src_offset) return MFSDP_ERR_OUT_OF_BOUNDS;
    if (g.dst_offset > dst_numel || g.numel > dst_numel - g.dst_offset) return MFSDP_ERR_OUT_OF_BOUNDS;
  }
  {
    std::vector<int> ord(n_segs);
    for (int i = 0; i < n_segs; ++i) ord[i] = i;
    std::sort(ord.begin(), ord.end(), [&](int x, int y) { return segs[x].dst_offset < segs[y].dst_offset; });
    for (int k = 1; k < n_segs; ++k)
      if (segs[ord[k - 1]].dst_offset + segs[ord[k - 1]].numel > segs[ord[k]].dst_offset) return MFSDP_ERR_OVERLAP;
  }
  // Chunk counts (2048 elements per CTA) must fit a launch grid.
  int64_t all_chunks = 0;
  for (int i = 0; i < n_segs; ++i) all_chunks += (segs[i].numel + kSegChunk - 1) / kSegChunk;
  if (all_chunks > (int64_t)INT32_MAX / 2) return MFSDP_ERR_UNSUPPORTED_SHAPE;

  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  for (int base = 0; base < n_segs; base += kMaxSegBatch) {
    const int cnt = std::min(kMaxSegBatch, n_segs - base);
    SegBatch b;
    std::memset(&b, 0, sizeof(b));
    b.n = cnt;
    b.mode = mode;
    b.n_src = n_src;
    b.src_bf16 = src_dtype == MFSDP_DTYPE_BF16;
    b.dst_bf16 = dst_dtype == MFSDP_DTYPE_BF16;
    b.dst = dst;
    for (int k = 0; k < n_src; ++k) b.src[k] = srcs[k];
    int64_t chunks = 0;
    for (int i = 0; i < cnt; ++i) {
      const mfsdp_segment& g = segs[base + i];
      b.seg[i].src_offset = g.src_offset;
      b.seg[i].dst_offset = g.dst_offset;
      b.seg[i].numel = g.numel;
      b.seg[i].src_index = g.src_index;
      b.chunk_start[i] = (int32_t)chunks;
      chunks += (g.numel + kSegChunk - 1) / kSegChunk;
    }
    b.chunk_start[cnt] = (int32_t)chunks;
    const PhaseRange range("mfsdp segment copy");
    const int st = cuda_status(launch_segments(b, (int)chunks, stream));
    if (st != MFSDP_OK) return st;
  }
  return MFSDP_OK;
}
