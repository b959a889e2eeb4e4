// Owner-shard checkpoints: one rank's optimizer state with the MatrixShard and
// tail tables that say where each parameter's state sits in its flat buffers.
//
// MatrixFSDP: Communication-Free Matrix Optimizers Under ZeRO-3 Parameter
// Sharding -- Abstract: the runtime carries the plan in MatrixShard metadata
// and supports owner-shard checkpoint resharding; FAQ (docshare page): the
// metadata carries the owner plan through optimizer routing and resharding.
// A file holds one rank's state; reloading under another world size re-plans,
// matches every parameter's old (owner, offset) to its new one
// (mfsdp_placement_segments) and copies it (mfsdp_segment_copy, GATHER).
//
// Layout, little-endian, independent of the host's byte order and struct
// padding (every field is written and read byte by byte):
//   "MFSDPCK1"                         8 bytes
//   format version (1)                 u32
//   world, rank, ns_steps              i32 x 3
//   n_matrix, n_tail                   i32 x 2
//   align_elems, matrix_elems,
//   tail_elems, adam_step              i64 x 4
//   n_matrix matrix shards             param_id i32, owner i32, offset i64,
//                                      rows i64, cols i64, transposed i32,
//                                      reserved i32, cost u64  (48 bytes each)
//   n_tail tail shards                 param_id i32, owner i32, offset i64,
//                                      numel i64  (24 bytes each)
//   momentum                           matrix_elems x f32 (IEEE binary32 bits)
//   tail p, m, v                       tail_elems x f32 each
//   FNV-1a 64 of every byte above      u64
#include <cstdio>
#include <cstring>
#include <vector>

#include "mfsdp.h"

namespace {

constexpr char kMagic[8] = {'M', 'F', 'S', 'D', 'P', 'C', 'K', '1'};
constexpr uint32_t kFormat = 1;
constexpr size_t kHeaderBytes = 8 + 4 + 3 * 4 + 2 * 4 + 4 * 8;
constexpr size_t kMatrixRecord = 48;
constexpr size_t kTailRecord = 24;

// FNV-1a, 64-bit (offset basis 14695981039346656037, prime 1099511628211).
struct Fnv {
  uint64_t h = 14695981039346656037ull;
  void add(const uint8_t* p, size_t n) {
    for (size_t i = 0; i < n; ++i) {
      h ^= p[i];
      h *= 1099511628211ull;
    }
  }
};

class Writer {
 public:
  explicit Writer(FILE* f) : f_(f) {}
  bool ok() const { return ok_; }
  uint64_t hash() const { return fnv_.h; }
  void bytes(const uint8_t* p, size_t n) {
    if (!ok_ || n == 0) return;
    fnv_.add(p, n);
    ok_ = std::fwrite(p, 1, n, f_) == n;
  }
  void u32(uint32_t v) {
    uint8_t b[4];
    for (int i = 0; i < 4; ++i) b[i] = (uint8_t)(v >> (8 * i));
    bytes(b, 4);
  }
  void u64(uint64_t v) {
    uint8_t b[8];
    for (int i = 0; i < 8; ++i) b[i] = (uint8_t)(v >> (8 * i));
    bytes(b, 8);
  }
  void i32(int32_t v) { u32((uint32_t)v); }
  void i64(int64_t v) { u64((uint64_t)v); }
  // n binary32 values, in chunks.
  void f32s(const float* p, int64_t n) {
    std::vector<uint8_t> buf;
    const int64_t chunk = 1 << 16;
    for (int64_t s = 0; s < n && ok_; s += chunk) {
      const int64_t c = n - s < chunk ? n - s : chunk;
      buf.resize((size_t)c * 4);
      for (int64_t i = 0; i < c; ++i) {
        uint32_t u;
        std::memcpy(&u, p + s + i, 4);
        for (int k = 0; k < 4; ++k) buf[(size_t)i * 4 + k] = (uint8_t)(u >> (8 * k));
      }
      bytes(buf.data(), buf.size());
    }
  }

 private:
  FILE* f_;
  bool ok_ = true;
  Fnv fnv_;
};

class Reader {
 public:
  explicit Reader(FILE* f) : f_(f) {}
  bool ok() const { return ok_; }
  uint64_t hash() const { return fnv_.h; }
  void bytes(uint8_t* p, size_t n) {
    if (!ok_ || n == 0) return;
    ok_ = std::fread(p, 1, n, f_) == n;
    if (ok_) fnv_.add(p, n);
  }
  uint32_t u32() {
    uint8_t b[4] = {0, 0, 0, 0};
    bytes(b, 4);
    uint32_t v = 0;
    for (int i = 0; i < 4; ++i) v |= (uint32_t)b[i] << (8 * i);
    return v;
  }
  uint64_t u64() {
    uint8_t b[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    bytes(b, 8);
    uint64_t v = 0;
    for (int i = 0; i < 8; ++i) v |= (uint64_t)b[i] << (8 * i);
    return v;
  }
  int32_t i32() { return (int32_t)u32(); }
  int64_t i64() { return (int64_t)u64(); }
  // n binary32 values into p, or skipped (hashed, not stored) when p is null.
  void f32s(float* p, int64_t n) {
    std::vector<uint8_t> buf;
    const int64_t chunk = 1 << 16;
    for (int64_t s = 0; s < n && ok_; s += chunk) {
      const int64_t c = n - s < chunk ? n - s : chunk;
      buf.resize((size_t)c * 4);
      bytes(buf.data(), buf.size());
      if (!ok_ || !p) continue;
      for (int64_t i = 0; i < c; ++i) {
        uint32_t u = 0;
        for (int k = 0; k < 4; ++k) u |= (uint32_t)buf[(size_t)i * 4 + k] << (8 * k);
        std::memcpy(p + s + i, &u, 4);
      }
    }
  }

 private:
  FILE* f_;
  bool ok_ = true;
  Fnv fnv_;
};

bool header_valid(const mfsdp_checkpoint_header& h) {
  return h.world >= 1 && h.rank >= 0 && h.rank < h.world && h.ns_steps >= 0 && h.n_matrix >= 0 && h.n_tail >= 0 &&
         h.align_elems >= 1 && h.matrix_elems >= 0 && h.tail_elems >= 0 && h.adam_step >= 0;
}

// Every shard of the rank's tables inside its buffers, owned by the rank.
bool tables_valid(const mfsdp_checkpoint_header& h, const mfsdp_matrix_shard* m, const mfsdp_tail_shard* t) {
  for (int32_t i = 0; i < h.n_matrix; ++i) {
    const mfsdp_matrix_shard& s = m[i];
    if (s.owner != h.rank || s.offset < 0 || s.rows < 1 || s.cols < 1 || s.rows > h.matrix_elems / s.cols ||
        s.offset > h.matrix_elems - s.rows * s.cols)
      return false;
  }
  for (int32_t i = 0; i < h.n_tail; ++i) {
    const mfsdp_tail_shard& s = t[i];
    if (s.owner != h.rank || s.offset < 0 || s.numel < 0 || s.offset > h.tail_elems - s.numel) return false;
  }
  return true;
}

int read_header(Reader& r, mfsdp_checkpoint_header* h) {
  char magic[8];
  r.bytes(reinterpret_cast<uint8_t*>(magic), 8);
  if (!r.ok()) return MFSDP_ERR_FORMAT;
  if (std::memcmp(magic, kMagic, 8) != 0) return MFSDP_ERR_FORMAT;
  const uint32_t version = r.u32();
  if (!r.ok() || version != kFormat) return MFSDP_ERR_FORMAT;
  h->world = r.i32();
  h->rank = r.i32();
  h->ns_steps = r.i32();
  h->n_matrix = r.i32();
  h->n_tail = r.i32();
  h->align_elems = r.i64();
  h->matrix_elems = r.i64();
  h->tail_elems = r.i64();
  h->adam_step = r.i64();
  if (!r.ok() || !header_valid(*h)) return MFSDP_ERR_FORMAT;
  return MFSDP_OK;
}

}  // namespace

extern "C" size_t mfsdp_checkpoint_bytes(const mfsdp_checkpoint_header* h) {
  if (!h || !header_valid(*h)) return 0;
  return kHeaderBytes + (size_t)h->n_matrix * kMatrixRecord + (size_t)h->n_tail * kTailRecord +
         4 * ((size_t)h->matrix_elems + 3 * (size_t)h->tail_elems) + 8;
}

extern "C" int mfsdp_checkpoint_write(const char* path, const mfsdp_checkpoint_header* h,
                                      const mfsdp_matrix_shard* matrix_shards, const mfsdp_tail_shard* tail_shards,
                                      const float* momentum, const float* tail_p, const float* tail_m,
                                      const float* tail_v) {
  if (!path || !h || !header_valid(*h)) return MFSDP_ERR_INVALID_ARG;
  if ((h->n_matrix > 0 && !matrix_shards) || (h->n_tail > 0 && !tail_shards)) return MFSDP_ERR_INVALID_ARG;
  if ((h->matrix_elems > 0 && !momentum) || (h->tail_elems > 0 && (!tail_p || !tail_m || !tail_v)))
    return MFSDP_ERR_INVALID_ARG;
  if (!tables_valid(*h, matrix_shards, tail_shards)) return MFSDP_ERR_OUT_OF_BOUNDS;
  FILE* f = std::fopen(path, "wb");
  if (!f) return MFSDP_ERR_IO;
  Writer w(f);
  w.bytes(reinterpret_cast<const uint8_t*>(kMagic), 8);
  w.u32(kFormat);
  w.i32(h->world);
  w.i32(h->rank);
  w.i32(h->ns_steps);
  w.i32(h->n_matrix);
  w.i32(h->n_tail);
  w.i64(h->align_elems);
  w.i64(h->matrix_elems);
  w.i64(h->tail_elems);
  w.i64(h->adam_step);
  for (int32_t i = 0; i < h->n_matrix; ++i) {
    const mfsdp_matrix_shard& s = matrix_shards[i];
    w.i32(s.param_id);
    w.i32(s.owner);
    w.i64(s.offset);
    w.i64(s.rows);
    w.i64(s.cols);
    w.i32(s.transposed);
    w.i32(s.reserved);
    w.u64(s.cost);
  }
  for (int32_t i = 0; i < h->n_tail; ++i) {
    const mfsdp_tail_shard& s = tail_shards[i];
    w.i32(s.param_id);
    w.i32(s.owner);
    w.i64(s.offset);
    w.i64(s.numel);
  }
  w.f32s(momentum, h->matrix_elems);
  w.f32s(tail_p, h->tail_elems);
  w.f32s(tail_m, h->tail_elems);
  w.f32s(tail_v, h->tail_elems);
  const uint64_t digest = w.hash();
  w.u64(digest);
  const bool ok = w.ok();
  const bool closed = std::fclose(f) == 0;
  return ok && closed ? MFSDP_OK : MFSDP_ERR_IO;
}

extern "C" int mfsdp_checkpoint_read_header(const char* path, mfsdp_checkpoint_header* h) {
  if (!path || !h) return MFSDP_ERR_INVALID_ARG;
  FILE* f = std::fopen(path, "rb");
  if (!f) return MFSDP_ERR_IO;
  Reader r(f);
  const int st = read_header(r, h);
  std::fclose(f);
  return st;
}

extern "C" int mfsdp_checkpoint_read(const char* path, mfsdp_checkpoint_header* h, mfsdp_matrix_shard* matrix_shards,
                                     int32_t matrix_capacity, mfsdp_tail_shard* tail_shards, int32_t tail_capacity,
                                     float* momentum, int64_t momentum_capacity, float* tail_p, float* tail_m,
                                     float* tail_v, int64_t tail_capacity_elems) {
  if (!path || !h) return MFSDP_ERR_INVALID_ARG;
  FILE* f = std::fopen(path, "rb");
  if (!f) return MFSDP_ERR_IO;
  Reader r(f);
  mfsdp_checkpoint_header hh;
  int st = read_header(r, &hh);
  if (st == MFSDP_OK) {
    if (hh.n_matrix > matrix_capacity || hh.n_tail > tail_capacity || hh.matrix_elems > momentum_capacity ||
        hh.tail_elems > tail_capacity_elems)
      st = MFSDP_ERR_WORKSPACE_TOO_SMALL;
    else if ((hh.n_matrix > 0 && !matrix_shards) || (hh.n_tail > 0 && !tail_shards) ||
             (hh.matrix_elems > 0 && !momentum) || (hh.tail_elems > 0 && (!tail_p || !tail_m || !tail_v)))
      st = MFSDP_ERR_INVALID_ARG;
  }
  if (st == MFSDP_OK) {
    for (int32_t i = 0; i < hh.n_matrix; ++i) {
      mfsdp_matrix_shard& s = matrix_shards[i];
      s.param_id = r.i32();
      s.owner = r.i32();
      s.offset = r.i64();
      s.rows = r.i64();
      s.cols = r.i64();
      s.transposed = r.i32();
      s.reserved = r.i32();
      s.cost = r.u64();
    }
    for (int32_t i = 0; i < hh.n_tail; ++i) {
      mfsdp_tail_shard& s = tail_shards[i];
      s.param_id = r.i32();
      s.owner = r.i32();
      s.offset = r.i64();
      s.numel = r.i64();
    }
    if (!r.ok() || !tables_valid(hh, matrix_shards, tail_shards)) st = MFSDP_ERR_FORMAT;
  }
  if (st == MFSDP_OK) {
    r.f32s(momentum, hh.matrix_elems);
    r.f32s(tail_p, hh.tail_elems);
    r.f32s(tail_m, hh.tail_elems);
    r.f32s(tail_v, hh.tail_elems);
    const uint64_t expect = r.hash();
    const uint64_t digest = r.u64();
    uint8_t extra;
    const bool at_end = std::fread(&extra, 1, 1, f) == 0;
    if (!r.ok() || digest != expect || !at_end) st = MFSDP_ERR_FORMAT;
  }
  std::fclose(f);
  if (st == MFSDP_OK) *h = hh;
  return st;
}
