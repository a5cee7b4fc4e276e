// Device buffer layouts shared by host and device code of libstp.so.
//
// tile_meta (caller-owned, written by stp_classify), for R rows of NT = T/128
// tiles, each array 256-byte aligned:
//   err        uint32                 device error word
//   cls        int8  [R][NT][NT]      0 EMPTY, 1 PARTIAL, 2 FULL (q-tile major)
//   csr_cnt    int32 [R][NT]          non-empty key tiles per query tile
//   csr        int32 [R][NT][NT]      (kt << 1) | partial, kt ascending
//   csc_cnt    int32 [R][NT]          non-empty query tiles per key tile
//   csc        int32 [R][NT][NT]      (qt << 1) | partial, qt ascending
//   kmin, kmax int32 [R][NT]          min / max subtree_end over each key tile
//
// fwd workspace: err (uint32) only.
// bwd workspace: err, delta float32 [R][Hq][T] (Delta on the float32 path,
// -Delta on the bf16 path), and for the bf16 path nlse2 float32 [R][Hq][T]
// (-LSE * log2 e) and dq_acc float32, one 128 x 128 tile per (row, query
// head, query tile), each tile stored [32 column quads][128 rows][4].
#pragma once

#include <cstddef>
#include <cstdint>

namespace stp {

constexpr int kTile = 128;
constexpr int kMaxRowLen = 131072;

enum : int8_t { kEmpty = 0, kPartial = 1, kFull = 2 };

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct TileMeta {
  size_t err, cls, csr_cnt, csr, csc_cnt, csc, kmin, kmax, total;
};

inline TileMeta tile_meta_layout(int64_t R, int64_t NT) {
  TileMeta m;
  size_t o = 0;
  m.err = o;     o += 256;
  m.cls = o;     o += align256(size_t(R * NT * NT));
  m.csr_cnt = o; o += align256(size_t(R * NT) * 4);
  m.csr = o;     o += align256(size_t(R * NT * NT) * 4);
  m.csc_cnt = o; o += align256(size_t(R * NT) * 4);
  m.csc = o;     o += align256(size_t(R * NT * NT) * 4);
  m.kmin = o;    o += align256(size_t(R * NT) * 4);
  m.kmax = o;    o += align256(size_t(R * NT) * 4);
  m.total = o;
  return m;
}

struct BwdWs {
  size_t err, delta, nlse2, dq_acc, total;
};

inline BwdWs bwd_ws_layout(int64_t R, int64_t T, int64_t Hq, int64_t D, bool need_acc) {
  BwdWs w;
  size_t o = 0;
  w.err = o;    o += 256;
  w.delta = o;  o += align256(size_t(R * Hq * T) * 4);
  w.nlse2 = o;  o += need_acc ? align256(size_t(R * Hq * T) * 4) : 0;
  w.dq_acc = o; o += need_acc ? align256(size_t(R * T * Hq * D) * 4) : 0;
  w.total = o;
  return w;
}

// Device error codes OR-ed into an error word.
enum : uint32_t {
  kErrBadSubtreeEnd = 1u << 0,  // subtree_end[j] outside [j, T)
  kErrTimeout = 1u << 1,        // a bounded wait ran out
  kErrBadList = 1u << 2,        // a tile list entry out of range
  kErrTmem = 1u << 3            // tensor-memory allocation returned an unusable address
};

}  // namespace stp
