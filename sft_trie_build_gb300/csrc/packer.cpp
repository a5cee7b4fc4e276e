// Host packer: global prefix tree, tree-aware best-fit-decreasing placement,
// materialization of packed rows.
//
// "Prefix tree packing" (furtherai.github.io/blog/posts/prefix-tree-packing):
//   tree-build section  -- longest agreed run emitted once, split by next token;
//                          minimum shared-segment length; trainable tokens are
//                          never shared; the join-token copy (placed where a
//                          member's next token is trainable, as the 32-rollout
//                          accounting fixes: "completion-length + 1" per rollout,
//                          the root paid in full);
//   global-tree section -- every sequence walks into one tree;
//   bin-packing section -- bins with occupied segments and a token count, the
//                          insertion delta, families ordered by their most
//                          expensive leaf, best fit with a strict test;
//   materialization     -- integers until the final single pass over tokens;
//   attention section   -- DFS enter/exit interval: row index = enter index,
//                          subtree_end = exit index.
//
// Shape of the implementation:
//   * the walk keeps an explicit stack instead of recursion; parts are pushed
//     in reverse so segments are numbered in DFS pre-order;
//   * a bin's occupied set is closed under ancestors (it is a union of
//     root-to-leaf paths), so the insertion delta is the length of the leaf's
//     path below its deepest occupied segment: walk up from the leaf and stop
//     at the first occupied segment;
//   * occupancy is one bitset per bin; exit indices come from one reverse
//     pass over the bin's segments in pre-order.
#include <algorithm>
#include <atomic>
#include <chrono>
#include <cstdio>
#include <cstring>
#include <new>
#include <mutex>
#include <string>
#include <system_error>
#include <thread>
#include <unordered_map>
#include <vector>

#include "internal.h"

namespace stp {

static thread_local std::string g_last_error;

stp_status fail(stp_status code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

void clear_error() { g_last_error.clear(); }

}  // namespace stp

using stp::fail;

namespace {

struct Segment {
  int32_t parent;  // -1 = root
  int64_t lo, hi;  // covered positions [lo, hi) of every member sequence
  int32_t rep;     // a member sequence (token source)
};

struct Bin {
  std::vector<int32_t> leaves;   // sequence ids in placement order
  std::vector<int32_t> segs;     // occupied segment ids (unsorted until finalize)
  std::vector<uint64_t> occ;     // occupancy bitset over segment ids
  int64_t tokens = 0;

  bool has(int32_t s) const { return (occ[s >> 6] >> (s & 63)) & 1ull; }
};

struct Walker {
  const int32_t* tok;
  const int64_t* off;
  const uint8_t* tr;
  int32_t min_shared;
  std::vector<int64_t> len, ntr;  // length and leading non-trainable count
  std::vector<Segment> segs;
  std::vector<int32_t> leaf_of;

  int32_t emit(int32_t parent, int64_t lo, int64_t hi, int32_t rep) {
    segs.push_back(Segment{parent, lo, hi, rep});
    return static_cast<int32_t>(segs.size() - 1);
  }
  int32_t token(int32_t s, int64_t p) const { return tok[off[s] + p]; }
  bool trainable_at(int32_t s, int64_t p) const { return tr && tr[off[s] + p]; }

  struct Work {
    std::vector<int32_t> members;  // ascending sequence ids
    int64_t start;
    int32_t parent;
  };

  // Split `members` at position p into ordered parts.  Sequences that end at p
  // or continue with a trainable token stand alone; the rest group by token.
  // Parts are ordered by (token at p, -1 if ended; smallest member id).
  void split(const std::vector<int32_t>& members, int64_t p,
             std::vector<std::vector<int32_t>>& parts) const {
    struct Part {
      int64_t key;
      int32_t first;
      std::vector<int32_t> m;
    };
    std::vector<Part> ps;
    std::unordered_map<int32_t, size_t> group_of;
    for (int32_t s : members) {
      if (len[s] == p) {
        ps.push_back(Part{-1, s, {s}});
      } else if (trainable_at(s, p)) {
        ps.push_back(Part{token(s, p), s, {s}});
      } else {
        int32_t t = token(s, p);
        auto it = group_of.find(t);
        if (it == group_of.end()) {
          group_of.emplace(t, ps.size());
          ps.push_back(Part{t, s, {s}});
        } else {
          ps[it->second].m.push_back(s);  // members arrive ascending
        }
      }
    }
    std::sort(ps.begin(), ps.end(), [](const Part& a, const Part& b) {
      return a.key != b.key ? a.key < b.key : a.first < b.first;
    });
    parts.clear();
    for (auto& q : ps) parts.push_back(std::move(q.m));
  }

  void walk(std::vector<int32_t> all) {
    std::vector<Work> stack;
    stack.push_back(Work{std::move(all), 0, -1});
    std::vector<std::vector<int32_t>> parts;
    while (!stack.empty()) {
      Work w = std::move(stack.back());
      stack.pop_back();
      const auto& S = w.members;
      if (S.size() == 1) {
        int32_t s = S[0];
        leaf_of[s] = emit(w.parent, w.start, len[s], s);
        continue;
      }
      // agreed run: every member non-trainable and equal on [start, start+A)
      int64_t lim = INT64_MAX;
      for (int32_t s : S) lim = std::min(lim, ntr[s]);
      int64_t A = std::max<int64_t>(0, lim - w.start);
      const int32_t* ref = tok + off[S[0]] + w.start;
      for (size_t k = 1; k < S.size() && A > 0; ++k) {
        const int32_t* o = tok + off[S[k]] + w.start;
        int64_t a = 0;
        while (a + 16 <= A && std::memcmp(o + a, ref + a, 16 * sizeof(int32_t)) == 0) a += 16;
        while (a < A && o[a] == ref[a]) ++a;
        A = a;
      }
      int64_t child_start;
      int32_t child_parent;
      int64_t split_at;
      if (A >= min_shared) {
        int64_t E = w.start + A;
        bool join = false;
        for (int32_t s : S) join = join || (ntr[s] == E && E < len[s]);
        int64_t seg_end = join ? E - 1 : E;
        child_parent = w.parent;
        if (seg_end > w.start) child_parent = emit(w.parent, w.start, seg_end, S[0]);
        child_start = seg_end;
        split_at = E;
      } else {
        child_start = w.start;
        child_parent = w.parent;
        split_at = w.start + A;
      }
      split(S, split_at, parts);
      for (size_t k = parts.size(); k-- > 0;)
        stack.push_back(Work{std::move(parts[k]), child_start, child_parent});
    }
  }
};

// Number of leading zero bytes of [p, p + n), eight bytes at a time.
int64_t leading_zero_bytes(const uint8_t* p, int64_t n) {
  int64_t k = 0;
  for (; k + 8 <= n; k += 8) {
    uint64_t w;
    std::memcpy(&w, p + k, 8);
    if (w) break;
  }
  while (k < n && !p[k]) ++k;
  return k;
}

}  // namespace

struct stp_plan {
  int32_t T = 0;
  int32_t min_shared = 0;
  uint32_t flags = 0;
  int32_t n_seqs = 0;
  std::vector<int32_t> tokens;
  std::vector<int64_t> offsets;
  std::vector<uint8_t> trainable;  // empty = none trainable
  std::vector<Segment> segs;
  std::vector<int32_t> leaf_of;
  std::vector<Bin> bins;
  std::vector<int32_t> row_of_seq;
  int64_t packed = 0;
  int64_t useful_pairs = 0;
  double walk_ms = 0.0;   // host wall time of the trie walk inside stp_pack
  double place_ms = 0.0;  // host wall time of the leaf placement inside stp_pack
};

namespace {

int64_t insertion_delta(const stp_plan& P, const Bin& b, int32_t leaf_seg) {
  int64_t d = 0;
  for (int32_t x = leaf_seg; x >= 0 && !b.has(x); x = P.segs[x].parent)
    d += P.segs[x].hi - P.segs[x].lo;
  return d;
}

void bin_add(stp_plan& P, Bin& b, int32_t seq) {
  for (int32_t x = P.leaf_of[seq]; x >= 0 && !b.has(x); x = P.segs[x].parent) {
    b.tokens += P.segs[x].hi - P.segs[x].lo;
    b.occ[x >> 6] |= 1ull << (x & 63);
    b.segs.push_back(x);
  }
  b.leaves.push_back(seq);
}

}  // namespace

extern "C" {

stp_status stp_pack(const int32_t* tokens, const int64_t* offsets, int32_t n_seqs,
                    const uint8_t* trainable, const int32_t* family, int32_t row_len,
                    int32_t min_shared, uint32_t flags, stp_plan** out) {
  stp::clear_error();
  if (!out) return fail(STP_EINVAL, "stp_pack: out is NULL");
  *out = nullptr;
  if (n_seqs < 0) return fail(STP_EINVAL, "stp_pack: n_seqs < 0");
  if (n_seqs > 0 && !offsets) return fail(STP_EINVAL, "stp_pack: offsets is NULL");
  if (row_len <= 0) return fail(STP_EINVAL, "stp_pack: row_len must be > 0");
  if (min_shared < 1) return fail(STP_EINVAL, "stp_pack: min_shared must be >= 1");
  if (flags & ~(uint32_t)(STP_PER_FAMILY | STP_IN_ORDER))
    return fail(STP_EINVAL, "stp_pack: unknown flag bits 0x%x", flags);
  if (n_seqs > 0 && offsets[0] != 0) return fail(STP_EINVAL, "stp_pack: offsets[0] != 0");
  for (int32_t s = 0; s < n_seqs; ++s) {
    if (offsets[s + 1] <= offsets[s])
      return fail(STP_EINVAL, "stp_pack: sequence %d is empty or offsets decrease", s);
  }
  int64_t total = n_seqs > 0 ? offsets[n_seqs] : 0;
  if (total > 0 && !tokens) return fail(STP_EINVAL, "stp_pack: tokens is NULL");
  for (int32_t s = 0; s < n_seqs; ++s) {
    if (offsets[s + 1] - offsets[s] > row_len)
      return fail(STP_ETOOLONG, "stp_pack: sequence %d has %lld tokens > row_len %d", s,
                  (long long)(offsets[s + 1] - offsets[s]), row_len);
  }

  stp_plan* P = new (std::nothrow) stp_plan();
  if (!P) return fail(STP_ENOMEM, "stp_pack: out of host memory");
  try {
    P->T = row_len;
    P->min_shared = min_shared;
    P->flags = flags;
    P->n_seqs = n_seqs;
    P->tokens.assign(tokens, tokens + total);
    P->offsets.assign(offsets, offsets + (n_seqs > 0 ? n_seqs + 1 : 0));
    if (trainable) P->trainable.assign(trainable, trainable + total);

    // families in order of first appearance
    std::vector<std::vector<int32_t>> fams;
    if (family) {
      std::unordered_map<int32_t, size_t> idx;
      for (int32_t s = 0; s < n_seqs; ++s) {
        auto it = idx.find(family[s]);
        if (it == idx.end()) {
          idx.emplace(family[s], fams.size());
          fams.push_back({s});
        } else {
          fams[it->second].push_back(s);
        }
      }
    } else {
      for (int32_t s = 0; s < n_seqs; ++s) fams.push_back({s});
    }

    using clock = std::chrono::steady_clock;
    const auto t_walk = clock::now();
    Walker w;
    w.tok = P->tokens.data();
    w.off = P->offsets.data();
    w.tr = P->trainable.empty() ? nullptr : P->trainable.data();
    w.min_shared = min_shared;
    w.len.resize(n_seqs);
    w.ntr.resize(n_seqs);
    w.leaf_of.assign(n_seqs, -1);
    for (int32_t s = 0; s < n_seqs; ++s) {
      w.len[s] = offsets[s + 1] - offsets[s];
      w.ntr[s] = w.tr ? leading_zero_bytes(w.tr + offsets[s], w.len[s]) : w.len[s];
    }
    if (n_seqs > 0) {
      if (flags & STP_PER_FAMILY) {
        for (auto& f : fams) {
          std::vector<int32_t> m(f);
          std::sort(m.begin(), m.end());
          w.walk(std::move(m));
        }
      } else {
        std::vector<int32_t> all(n_seqs);
        for (int32_t s = 0; s < n_seqs; ++s) all[s] = s;
        w.walk(std::move(all));
      }
    }
    P->segs = std::move(w.segs);
    P->leaf_of = std::move(w.leaf_of);
    const auto t_place = clock::now();
    P->walk_ms = std::chrono::duration<double, std::milli>(t_place - t_walk).count();

    const size_t words = (P->segs.size() + 63) / 64;
    auto new_bin = [&]() -> Bin& {
      P->bins.emplace_back();
      P->bins.back().occ.assign(words, 0);
      return P->bins.back();
    };
    if (flags & STP_IN_ORDER) {
      for (int32_t s = 0; s < n_seqs; ++s) {
        if (P->bins.empty() ||
            P->bins.back().tokens + insertion_delta(*P, P->bins.back(), P->leaf_of[s]) > row_len)
          new_bin();
        bin_add(*P, P->bins.back(), s);
      }
    } else {
      // families by their most expensive leaf, descending, stable
      std::vector<std::pair<int64_t, size_t>> order;
      for (size_t f = 0; f < fams.size(); ++f) {
        int64_t mx = 0;
        for (int32_t s : fams[f]) mx = std::max(mx, w.len[s]);
        order.emplace_back(mx, f);
      }
      std::stable_sort(order.begin(), order.end(),
                       [](const auto& a, const auto& b) { return a.first > b.first; });
      for (auto& of : order) {
        for (int32_t s : fams[of.second]) {
          int32_t leaf = P->leaf_of[s];
          int64_t best_room = (int64_t)row_len + 1;
          long best = -1;
          for (size_t b = 0; b < P->bins.size(); ++b) {
            int64_t count = P->bins[b].tokens + insertion_delta(*P, P->bins[b], leaf);
            if (count <= row_len && row_len - count < best_room) {
              best_room = row_len - count;
              best = (long)b;
            }
          }
          if (best < 0) {
            new_bin();
            best = (long)P->bins.size() - 1;
          }
          bin_add(*P, P->bins[best], s);
        }
      }
    }
    P->place_ms = std::chrono::duration<double, std::milli>(clock::now() - t_place).count();
    P->row_of_seq.assign(n_seqs, -1);
    for (size_t b = 0; b < P->bins.size(); ++b) {
      Bin& bn = P->bins[b];
      std::sort(bn.segs.begin(), bn.segs.end());
      P->packed += bn.tokens;
      for (int32_t s : bn.leaves) P->row_of_seq[s] = (int32_t)b;
      for (int32_t x : bn.segs) {
        // sum over covered positions p of (p + 1)
        int64_t lo = P->segs[x].lo, hi = P->segs[x].hi;
        P->useful_pairs += (hi * (hi + 1) - lo * (lo + 1)) / 2;
      }
    }
  } catch (const std::bad_alloc&) {
    delete P;
    return fail(STP_ENOMEM, "stp_pack: out of host memory");
  }
  *out = P;
  return STP_OK;
}

stp_status stp_plan_info(const stp_plan* P, stp_plan_info_t* info) {
  stp::clear_error();
  if (!P || !info) return fail(STP_EINVAL, "stp_plan_info: NULL argument");
  info->n_rows = (int32_t)P->bins.size();
  info->row_len = P->T;
  info->input_tokens = P->tokens.size();
  info->packed_tokens = P->packed;
  info->n_segments = (int64_t)P->segs.size();
  info->n_leaves = P->n_seqs;
  info->useful_pairs = P->useful_pairs;
  info->tree_token_ratio = P->packed ? (double)P->tokens.size() / (double)P->packed : 0.0;
  return STP_OK;
}

stp_status stp_plan_times(const stp_plan* P, double* walk_ms, double* place_ms) {
  stp::clear_error();
  if (!P || !walk_ms || !place_ms) return fail(STP_EINVAL, "stp_plan_times: NULL argument");
  *walk_ms = P->walk_ms;
  *place_ms = P->place_ms;
  return STP_OK;
}

stp_status stp_plan_rows_of(const stp_plan* P, int32_t* row_of_seq) {
  stp::clear_error();
  if (!P || (!row_of_seq && P->n_seqs > 0)) return fail(STP_EINVAL, "stp_plan_rows_of: NULL argument");
  std::copy(P->row_of_seq.begin(), P->row_of_seq.end(), row_of_seq);
  return STP_OK;
}

stp_status stp_plan_write(const stp_plan* P, int32_t* token_ids, int32_t* position_ids,
                          int32_t* subtree_end, uint8_t* loss_mask, int64_t* gather_index) {
  stp::clear_error();
  if (!P) return fail(STP_EINVAL, "stp_plan_write: plan is NULL");
  const int64_t T = P->T;
  const size_t nseg = P->segs.size();
  std::vector<int64_t> start(nseg, -1), last(nseg, -1);
  std::vector<uint8_t> is_leaf(nseg, 0);
  for (int32_t x : P->leaf_of) is_leaf[x] = 1;
  const uint8_t* tr = P->trainable.empty() ? nullptr : P->trainable.data();
  for (size_t r = 0; r < P->bins.size(); ++r) {
    const Bin& b = P->bins[r];
    const int64_t base = (int64_t)r * T;
    int64_t cur = 0;
    for (int32_t x : b.segs) {
      const Segment& sg = P->segs[x];
      const int64_t n = sg.hi - sg.lo;
      start[x] = cur;
      last[x] = n > 0 ? cur + n - 1 : -1;
      if (token_ids && n > 0)
        std::memcpy(token_ids + base + cur, P->tokens.data() + P->offsets[sg.rep] + sg.lo, n * sizeof(int32_t));
      if (position_ids)
        for (int64_t k = 0; k < n; ++k) position_ids[base + cur + k] = (int32_t)(sg.lo + k);
      cur += n;
    }
    // exit index: children follow their parent in pre-order, so one reverse
    // pass carries every subtree's last row index up to its ancestors
    for (size_t k = b.segs.size(); k-- > 0;) {
      int32_t x = b.segs[k];
      int32_t p = P->segs[x].parent;
      if (p >= 0 && last[x] >= 0) last[p] = std::max(last[p], last[x]);
    }
    if (subtree_end) {
      for (int32_t x : b.segs) {
        const int64_t n = P->segs[x].hi - P->segs[x].lo;
        std::fill(subtree_end + base + start[x], subtree_end + base + start[x] + n, (int32_t)last[x]);
      }
      for (int64_t j = cur; j < T; ++j) subtree_end[base + j] = (int32_t)j;
    }
    if (token_ids) std::fill(token_ids + base + cur, token_ids + base + T, 0);
    if (position_ids) std::fill(position_ids + base + cur, position_ids + base + T, 0);
    if (loss_mask) std::memset(loss_mask + base, 0, (size_t)T);
    for (int32_t s : b.leaves) {
      const int64_t o = P->offsets[s], L = P->offsets[s + 1] - o;
      for (int32_t x = P->leaf_of[s]; x >= 0; x = P->segs[x].parent) {
        const Segment& sg = P->segs[x];
        const int64_t flat0 = base + start[x] - sg.lo;  // row-major index of position p is flat0 + p
        if (gather_index)
          for (int64_t p = sg.lo; p < sg.hi; ++p) gather_index[o + p] = flat0 + p;
        // a loss position is one whose next token is trainable; the walk ends
        // every shared segment before a trainable token, so only the leaf's
        // own segment can hold one
        if (loss_mask && tr && is_leaf[x]) {
          const int64_t hi = std::min<int64_t>(sg.hi, L - 1);
          for (int64_t p = sg.lo; p < hi; ++p)
            if (tr[o + p + 1]) loss_mask[flat0 + p] = 1;
        }
      }
    }
  }
  return STP_OK;
}

void stp_plan_free(stp_plan* P) { delete P; }

}  // extern "C"

// ---------------------------------------------------------------------------
// "What if" planning: rows a candidate batch would need ("Prefix tree packing",
// global-tree section: the same tree-and-bin-pack pass that packs a step is
// run over sampled subsets of past data to estimate the rows of a candidate
// batch before committing to it).  A subset is gathered into contiguous
// arrays and planned by stp_pack itself, so the count is exactly what packing
// that batch would give; nothing is materialized.
// ---------------------------------------------------------------------------

namespace {

stp_status plan_rows_one(const int32_t* tokens, const int64_t* offsets, int32_t n_seqs,
                         const uint8_t* trainable, const int32_t* family, const int32_t* subset,
                         int32_t n_subset, int32_t row_len, int32_t min_shared, uint32_t flags,
                         int32_t* n_rows, int64_t* packed) {
  std::vector<int32_t> t2, f2;
  std::vector<int64_t> o2;
  std::vector<uint8_t> tr2;
  const int32_t *tk = tokens, *fm = family;
  const int64_t* of = offsets;
  const uint8_t* tr = trainable;
  int32_t n = n_seqs;
  if (subset) {
    int64_t total = 0;
    for (int32_t i = 0; i < n_subset; ++i) {
      const int32_t s = subset[i];
      if (s < 0 || s >= n_seqs) return fail(STP_EINVAL, "subset[%d] = %d outside [0, %d)", i, s, n_seqs);
      total += offsets[s + 1] - offsets[s];
    }
    try {
      t2.reserve(total);
      o2.reserve(n_subset + 1);
      o2.push_back(0);
      if (trainable) tr2.reserve(total);
      if (family) f2.reserve(n_subset);
      for (int32_t i = 0; i < n_subset; ++i) {
        const int32_t s = subset[i];
        t2.insert(t2.end(), tokens + offsets[s], tokens + offsets[s + 1]);
        if (trainable) tr2.insert(tr2.end(), trainable + offsets[s], trainable + offsets[s + 1]);
        if (family) f2.push_back(family[s]);
        o2.push_back((int64_t)t2.size());
      }
    } catch (const std::bad_alloc&) {
      return fail(STP_ENOMEM, "out of host memory");
    }
    tk = t2.data();
    of = o2.data();
    tr = trainable ? tr2.data() : nullptr;
    fm = family ? f2.data() : nullptr;
    n = n_subset;
  }
  stp_plan* P = nullptr;
  const stp_status st = stp_pack(tk, of, n, tr, fm, row_len, min_shared, flags, &P);
  if (st) return st;
  *n_rows = (int32_t)P->bins.size();
  *packed = P->packed;
  stp_plan_free(P);
  return STP_OK;
}

}  // namespace

extern "C" {

stp_status stp_plan_rows(const int32_t* tokens, const int64_t* offsets, int32_t n_seqs,
                         const uint8_t* trainable, const int32_t* family, const int32_t* subset,
                         int32_t n_subset, int32_t row_len, int32_t min_shared, uint32_t flags,
                         int32_t* n_rows, int64_t* packed_tokens) {
  stp::clear_error();
  if (!n_rows || !packed_tokens) return fail(STP_EINVAL, "stp_plan_rows: NULL output");
  if (n_seqs < 0 || n_subset < 0) return fail(STP_EINVAL, "stp_plan_rows: negative count");
  if (n_seqs > 0 && !offsets) return fail(STP_EINVAL, "stp_plan_rows: offsets is NULL");
  return plan_rows_one(tokens, offsets, n_seqs, trainable, family, subset, n_subset, row_len,
                       min_shared, flags, n_rows, packed_tokens);
}

stp_status stp_plan_rows_many(const int32_t* tokens, const int64_t* offsets, int32_t n_seqs,
                              const uint8_t* trainable, const int32_t* family,
                              const int32_t* subsets, const int64_t* subset_offsets,
                              int32_t n_subsets, int32_t row_len, int32_t min_shared,
                              uint32_t flags, int32_t n_threads, int32_t* n_rows,
                              int64_t* packed_tokens) {
  stp::clear_error();
  if (n_subsets < 0 || n_seqs < 0) return fail(STP_EINVAL, "stp_plan_rows_many: negative count");
  if (n_subsets == 0) return STP_OK;
  if (!subsets || !subset_offsets || !n_rows || !packed_tokens)
    return fail(STP_EINVAL, "stp_plan_rows_many: NULL argument");
  if (n_seqs > 0 && !offsets) return fail(STP_EINVAL, "stp_plan_rows_many: offsets is NULL");
  if (subset_offsets[0] != 0) return fail(STP_EINVAL, "stp_plan_rows_many: subset_offsets[0] != 0");
  for (int32_t i = 0; i < n_subsets; ++i)
    if (subset_offsets[i + 1] < subset_offsets[i] || subset_offsets[i + 1] - subset_offsets[i] > INT32_MAX)
      return fail(STP_EINVAL, "stp_plan_rows_many: subset_offsets decrease at %d", i);
  int nt = n_threads > 0 ? n_threads : (int)std::thread::hardware_concurrency();
  nt = std::max(1, std::min(nt, (int)n_subsets));
  std::atomic<int32_t> next{0};
  std::mutex mu;
  stp_status first = STP_OK;
  std::string msg;
  auto work = [&]() {
    for (int32_t i = next++; i < n_subsets; i = next++) {
      const int64_t a = subset_offsets[i], b = subset_offsets[i + 1];
      const stp_status st = plan_rows_one(tokens, offsets, n_seqs, trainable, family, subsets + a,
                                          (int32_t)(b - a), row_len, min_shared, flags, n_rows + i,
                                          packed_tokens + i);
      if (st) {
        std::lock_guard<std::mutex> lock(mu);
        if (!first) {
          first = st;
          msg = "subset " + std::to_string(i) + ": " + stp_last_error();
        }
      }
    }
  };
  try {
    std::vector<std::thread> pool;
    for (int t = 1; t < nt; ++t) pool.emplace_back(work);
    work();
    for (auto& th : pool) th.join();
  } catch (const std::system_error&) {
    return fail(STP_ENOMEM, "stp_plan_rows_many: cannot start host threads");
  }
  if (first) return fail(first, "stp_plan_rows_many: %s", msg.c_str());
  return STP_OK;
}

const char* stp_last_error(void) { return stp::g_last_error.c_str(); }

const char* stp_version(void) { return "stp 0.1 (sm_103a)"; }

}  // extern "C"
