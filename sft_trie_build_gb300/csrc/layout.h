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
//   crank      int32 [R][NT][NT]      crank[r][qt][kt]: position of kt in the
//                                     csr list of qt (set for non-empty pairs)
//   csr_off    int32 [R][NT]          non-empty pairs of the row before query tile qt
//   row_base   int32 [R]              first pair index of the row
//   csc_pair   int32 [R][NT][NT]      pair index of each csc entry
//   pair_count int32                  non-empty pairs over all rows
// A non-empty (query tile, key tile) pair has the index
// row_base[r] + csr_off[r][qt] + (position of kt in the csr list of qt):
// pairs are numbered query-tile major, key tiles ascending, rows in any order.
//
// fwd workspace: err (uint32) only.
// bwd workspace: err; on the float32 path delta float32 [R][Hq][T]; on the
// bf16 path two bias tiles per (row, head, query tile), sbias and dbias
// [R][Hq][NT] x 4 KiB (the row bias -LSE / scale of the scores and -Delta of
// dP, each split into three bf16 terms, laid out as the B operand of one
// K = 16 MMA: see bwd_delta_kernel), and ds: `slots` slots, each holding one bf16 128 x 128
// tile of dS^T per (pair, query head of one kv-head group), pair-major; a
// tile is 16 blocks of 2048 bytes, block c holding query columns 8c..8c+7 of
// the 128 keys, 16 bytes per key.  The backward runs its kv heads in at most
// kBwdGroups groups; a slot serves one group at a time.
#pragma once

#include <cstddef>
#include <cstdint>

namespace stp {

constexpr int kTile = 128;
constexpr int kMaxRowLen = 131072;

enum : int8_t { kEmpty = 0, kPartial = 1, kFull = 2 };

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct TileMeta {
  size_t err, cls, csr_cnt, csr, csc_cnt, csc, kmin, kmax, crank, csr_off, row_base, csc_pair,
      pair_count, total;
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
  m.crank = o;   o += align256(size_t(R * NT * NT) * 4);
  m.csr_off = o; o += align256(size_t(R * NT) * 4);
  m.row_base = o; o += align256(size_t(R) * 4);
  m.csc_pair = o; o += align256(size_t(R * NT * NT) * 4);
  m.pair_count = o; o += 256;
  m.total = o;
  return m;
}

constexpr size_t kDsTileBytes = 128 * 128 * 2;  // one bf16 dS^T tile

// Gated DeltaNet: tokens per chunk of the chunked recurrence, and the layout
// of the host plan (int32 words; a header of kGdnHeader words, then arrays).
constexpr int kGdnChunk = 64;
// A root segment of at least kGdnSplitChunks chunks is planned as two: its
// first kGdnHeadChunks chunks (depth 0), then the rest as their only child,
// so that the first walk starts after a short preparation and the rest is
// prepared beside it.  The cut falls on a chunk boundary: every chunk, and
// so every result, is the same as without it.
constexpr int kGdnHeadChunks = 16;
constexpr int kGdnSplitChunks = 32;
constexpr int kGdnHeader = 24;
constexpr int32_t kGdnMagic = 0x31444e47;  // "GDN1"
enum GdnPlanField {
  GP_MAGIC = 0, GP_N, GP_NSEG, GP_NCHUNK, GP_NDEPTH, GP_WORDS, GP_PREV, GP_SEG_START, GP_SEG_LEN,
  GP_SEG_PARENT, GP_SEG_CHUNK0, GP_DEPTH_OFF, GP_CHUNK_START, GP_CHUNK_LEN, GP_MAX_DEPTH_SEGS, GP_PREV2, GP_PREV3,
  GP_CHILD_OFF, GP_CHILD, GP_SUCC_OFF, GP_SUCC
};

// Non-empty pairs the dS workspace holds: the descriptor's max_tile_pairs, or
// when that is 0 every pair with kt <= qt (R NT (NT+1) / 2).
inline int64_t pair_capacity(int64_t R, int64_t NT, int64_t max_tile_pairs) {
  return max_tile_pairs > 0 ? max_tile_pairs : R * NT * (NT + 1) / 2;
}

// Groups of whole kv heads of one backward call (each launched on its own
// stream): n = min(Hkv, kBwdGroups) groups, group i holding kv heads
// [i Hkv / n, (i + 1) Hkv / n); `group_heads` query heads at most per group.
constexpr int kBwdGroups = 8;
struct BwdGroups {
  int n, group_heads, slots;
};
inline BwdGroups bwd_groups(int Hq, int Hkv, int ds_groups) {
  BwdGroups b;
  b.n = Hkv < kBwdGroups ? Hkv : kBwdGroups;
  b.group_heads = ((Hkv + b.n - 1) / b.n) * (Hq / Hkv);
  b.slots = (ds_groups <= 0 || ds_groups > b.n) ? b.n : ds_groups;
  return b;
}

constexpr size_t kBiasTileBytes = 4096;  // one query tile's bias: 128 queries x 16 bf16

struct BwdWs {
  size_t err, delta, sbias, dbias, ds, slot_bytes, total;
};

inline BwdWs bwd_ws_layout(int64_t R, int64_t T, int64_t Hq, int64_t Hkv, bool tensor_path, int64_t cap_pairs,
                           int ds_groups) {
  BwdWs w;
  const BwdGroups b = bwd_groups((int)Hq, (int)Hkv, ds_groups);
  size_t o = 0;
  const size_t bias = size_t(R * Hq * (T / kTile)) * kBiasTileBytes;
  w.err = o;    o += 256;
  w.delta = o;  o += tensor_path ? 0 : align256(size_t(R * Hq * T) * 4);
  w.sbias = o;  o += tensor_path ? bias : 0;
  w.dbias = o;  o += tensor_path ? bias : 0;
  w.slot_bytes = size_t(cap_pairs) * size_t(b.group_heads) * kDsTileBytes;
  w.ds = o;     o += tensor_path ? size_t(b.slots) * w.slot_bytes : 0;
  w.total = o;
  return w;
}

// Device error codes OR-ed into an error word.
enum : uint32_t {
  kErrBadSubtreeEnd = 1u << 0,  // subtree_end[j] outside [j, T)
  kErrTimeout = 1u << 1,        // a bounded wait ran out
  kErrBadList = 1u << 2,        // a tile list entry out of range
  kErrTmem = 1u << 3,           // tensor-memory allocation returned an unusable address
  kErrCapacity = 1u << 4        // more non-empty tile pairs than the dS workspace holds
};

}  // namespace stp
