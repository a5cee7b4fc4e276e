// Host planner of the tree-aware Gated DeltaNet ("Prefix tree packing", GDN
// section: the state is threaded along each path, forked at every branch
// point and zero at every root; the planner walks the tree depth by depth and
// coalesces all segments of one depth into one pass).
//
// From subtree_end alone: the token before x on its path is the nearest
// earlier token whose subtree still holds x (a stack over the DFS order).  A
// segment is a maximal run x, x + 1, ... in which every token continues the
// previous one and the previous one has no other child; a branch point
// therefore always ends its segment, and every segment starts from the final
// state of its parent segment.  A root segment of at least kGdnSplitChunks
// chunks is cut after its first kGdnHeadChunks chunks into two segments, the
// second the only child of the first (chunk for chunk the same work; the
// forward then walks the first while it prepares the rest).  Segments are
// sorted by depth (stable) and cut into chunks of kGdnChunk tokens, the last
// one ragged.
#include <cstring>
#include <vector>

#include "internal.h"
#include "layout.h"

using namespace stp;

namespace {

stp_status check_gdn(const stp_gdn_desc* d) {
  if (!d) return fail(STP_EINVAL, "GDN descriptor is NULL");
  if (d->n_rows < 0 || d->row_len <= 0 || d->row_len > kMaxRowLen)
    return fail(STP_EINVAL, "need n_rows >= 0 and row_len in [1, %d]", kMaxRowLen);
  if ((int64_t)d->n_rows * d->row_len > (1 << 26)) return fail(STP_EUNSUPPORTED, "more than 2^26 tokens");
  return STP_OK;
}

}  // namespace

extern "C" stp_status stp_gdn_plan_bound(const stp_gdn_desc* desc, size_t* plan_bytes) {
  clear_error();
  stp_status st = check_gdn(desc);
  if (st) return st;
  if (!plan_bytes) return fail(STP_EINVAL, "stp_gdn_plan_bound: NULL output");
  const size_t N = (size_t)desc->n_rows * desc->row_len;
  // prev (1, 2 and 3 back), 4 words per segment, depth offsets, 2 words per chunk, the child lists
  // (segments, chunks <= N), the token successor lists
  *plan_bytes = 4 * (kGdnHeader + 3 * N + 4 * N + (N + 1) + 2 * N + (N + 1) + N + (N + 1) + N);
  return STP_OK;
}

extern "C" stp_status stp_gdn_plan(const stp_gdn_desc* desc, const int32_t* subtree_end, const int32_t* row_used,
                                   void* plan, size_t plan_bytes) {
  clear_error();
  stp_status st = check_gdn(desc);
  if (st) return st;
  if (!subtree_end || !plan) return fail(STP_EINVAL, "stp_gdn_plan: NULL pointer");
  const int R = desc->n_rows, T = desc->row_len;
  const int64_t N = (int64_t)R * T;
  size_t bound = 0;
  stp_gdn_plan_bound(desc, &bound);
  if (plan_bytes < bound) return fail(STP_EINVAL, "stp_gdn_plan: plan buffer of %zu bytes, need %zu", plan_bytes, bound);

  std::vector<int32_t> prev(N, -2), n_child(N, 0);
  std::vector<int32_t> stack;
  for (int r = 0; r < R; ++r) {
    const int used = row_used ? row_used[r] : T;
    if (used < 0 || used > T) return fail(STP_EINVAL, "row_used[%d] = %d outside [0, %d]", r, used, T);
    const int32_t* se = subtree_end + (int64_t)r * T;
    const int64_t base = (int64_t)r * T;
    stack.clear();
    for (int x = 0; x < used; ++x) {
      if (se[x] < x || se[x] >= T) return fail(STP_EINVAL, "subtree_end[%d][%d] = %d outside [x, T)", r, x, se[x]);
      while (!stack.empty() && se[stack.back()] < x) stack.pop_back();
      if (!stack.empty()) {
        const int p = stack.back();
        if (se[x] > se[p])
          return fail(STP_EINVAL, "subtree_end[%d][%d] = %d leaves the subtree of its parent %d", r, x, se[x], p);
        prev[base + x] = (int32_t)(base + p);
        ++n_child[base + p];
      } else {
        prev[base + x] = -1;
      }
      stack.push_back(x);
    }
  }

  // x continues the run of x - 1 (same row, x - 1's only child)
  auto continues = [&](int64_t x) { return prev[x] == x - 1 && x % T != 0 && n_child[x - 1] == 1; };
  // where long root runs are cut: kGdnHeadChunks chunks after their first token
  std::vector<char> cut(N, 0);
  for (int64_t x = 0; x < N; ++x) {
    if (prev[x] != -1) continue;
    int64_t y = x + 1;
    while (y < N && continues(y)) ++y;
    if (y - x >= (int64_t)kGdnSplitChunks * kGdnChunk) cut[x + (int64_t)kGdnHeadChunks * kGdnChunk] = 1;
    x = y - 1;
  }

  // segments in token (DFS) order: parents come before their children
  std::vector<int64_t> s_start;
  std::vector<int32_t> s_len, s_parent, s_depth, seg_of(N, -1);
  for (int64_t x = 0; x < N; ++x) {
    if (prev[x] == -2) continue;
    const bool cont = continues(x) && !cut[x];
    if (!cont) {
      const int32_t par = prev[x] >= 0 ? seg_of[prev[x]] : -1;
      s_start.push_back(x);
      s_len.push_back(0);
      s_parent.push_back(par);
      s_depth.push_back(par >= 0 ? s_depth[par] + 1 : 0);
    }
    seg_of[x] = (int32_t)(s_start.size() - 1);
    ++s_len.back();
  }
  const int32_t n_seg = (int32_t)s_start.size();
  int32_t n_depth = 0;
  for (int32_t d : s_depth) n_depth = d + 1 > n_depth ? d + 1 : n_depth;

  // stable counting sort by depth; new index of each segment
  std::vector<int32_t> depth_off(n_depth + 1, 0), order(n_seg), new_of(n_seg);
  for (int32_t d : s_depth) ++depth_off[d + 1];
  int32_t max_depth_segs = 0;
  for (int d = 0; d < n_depth; ++d) {
    max_depth_segs = depth_off[d + 1] > max_depth_segs ? depth_off[d + 1] : max_depth_segs;
    depth_off[d + 1] += depth_off[d];
  }
  {
    std::vector<int32_t> fill(depth_off.begin(), depth_off.end() - 1);
    for (int32_t s = 0; s < n_seg; ++s) {
      new_of[s] = fill[s_depth[s]]++;
      order[new_of[s]] = s;
    }
  }
  int32_t n_chunk = 0;
  for (int32_t s = 0; s < n_seg; ++s) n_chunk += (s_len[s] + kGdnChunk - 1) / kGdnChunk;

  int32_t* w = static_cast<int32_t*>(plan);
  std::memset(w, 0, 4 * kGdnHeader);
  int64_t o = kGdnHeader;
  auto take = [&](int field, int64_t n) {
    w[field] = (int32_t)o;
    o += n;
  };
  take(GP_PREV, N);
  take(GP_PREV2, N);
  take(GP_PREV3, N);
  take(GP_SEG_START, n_seg);
  take(GP_SEG_LEN, n_seg);
  take(GP_SEG_PARENT, n_seg);
  take(GP_SEG_CHUNK0, n_seg);
  take(GP_DEPTH_OFF, n_depth + 1);
  take(GP_CHUNK_START, n_chunk);
  take(GP_CHUNK_LEN, n_chunk);
  take(GP_CHILD_OFF, n_seg + 1);
  take(GP_CHILD, n_seg);
  int64_t n_succ = 0;
  for (int64_t x = 0; x < N; ++x) n_succ += prev[x] >= 0;
  take(GP_SUCC_OFF, N + 1);
  take(GP_SUCC, n_succ);
  w[GP_MAGIC] = kGdnMagic;
  w[GP_N] = (int32_t)N;
  w[GP_NSEG] = n_seg;
  w[GP_NCHUNK] = n_chunk;
  w[GP_NDEPTH] = n_depth;
  w[GP_WORDS] = (int32_t)o;
  w[GP_MAX_DEPTH_SEGS] = max_depth_segs;
  std::memcpy(w + w[GP_PREV], prev.data(), 4 * N);
  for (int64_t x = 0; x < N; ++x) {   // two and three tokens back on the path (-1: none)
    const int32_t p1 = prev[x], p2 = p1 >= 0 ? prev[p1] : -1;
    w[w[GP_PREV2] + x] = p2;
    w[w[GP_PREV3] + x] = p2 >= 0 ? prev[p2] : -1;
  }
  int32_t c = 0;
  for (int32_t i = 0; i < n_seg; ++i) {
    const int32_t s = order[i];
    w[w[GP_SEG_START] + i] = (int32_t)s_start[s];
    w[w[GP_SEG_LEN] + i] = s_len[s];
    w[w[GP_SEG_PARENT] + i] = s_parent[s] >= 0 ? new_of[s_parent[s]] : -1;
    w[w[GP_SEG_CHUNK0] + i] = c;
    for (int32_t a = 0; a < s_len[s]; a += kGdnChunk, ++c) {
      w[w[GP_CHUNK_START] + c] = (int32_t)(s_start[s] + a);
      w[w[GP_CHUNK_LEN] + c] = s_len[s] - a < kGdnChunk ? s_len[s] - a : kGdnChunk;
    }
  }
  for (int d = 0; d <= n_depth; ++d) w[w[GP_DEPTH_OFF] + d] = depth_off[d];
  // children of each (sorted) segment, as a CSR list in the sorted numbering
  {
    int32_t* off = w + w[GP_CHILD_OFF];
    int32_t* ch = w + w[GP_CHILD];
    for (int32_t i = 0; i <= n_seg; ++i) off[i] = 0;
    for (int32_t i = 0; i < n_seg; ++i) {
      const int32_t par = w[w[GP_SEG_PARENT] + i];
      if (par >= 0) ++off[par + 1];
    }
    for (int32_t i = 0; i < n_seg; ++i) off[i + 1] += off[i];
    std::vector<int32_t> fill(off, off + n_seg);
    for (int32_t i = 0; i < n_seg; ++i) {
      const int32_t par = w[w[GP_SEG_PARENT] + i];
      if (par >= 0) ch[fill[par]++] = i;
    }
  }
  // successors of every token (the tokens whose path predecessor it is), in
  // token order, as a CSR list: the convolution's input gradient of a token
  // gathers from them
  {
    int32_t* off = w + w[GP_SUCC_OFF];
    int32_t* sc = w + w[GP_SUCC];
    for (int64_t x = 0; x <= N; ++x) off[x] = 0;
    for (int64_t x = 0; x < N; ++x)
      if (prev[x] >= 0) ++off[prev[x] + 1];
    for (int64_t x = 0; x < N; ++x) off[x + 1] += off[x];
    std::vector<int32_t> fill(off, off + N);
    for (int64_t x = 0; x < N; ++x)
      if (prev[x] >= 0) sc[fill[prev[x]]++] = (int32_t)x;
  }
  return STP_OK;
}
