// Tile classification of packed rows ("Prefix tree packing", attention
// section: a token's visible set is one fully visible block per ancestor
// segment plus a causal triangle over its own segment; most blocks of a
// packed row are empty and are skipped).
//
// With the interval predicate  visible(i, j) <=> j <= i && se[j] >= i  and
// se[j] >= j, a (query tile [q0,q1), key tile [k0,k1)) pair is
//   FULL    iff k1 - 1 <= q0 and min_{j in tile} se[j] >= q1 - 1,
//   EMPTY   iff k0 > q1 - 1 or max_{j in [k0, min(k1,q1))} se[j] < q0,
//   PARTIAL otherwise.
// For 128-aligned tiles this reduces to: kt > qt EMPTY, kt == qt PARTIAL
// (i = j is always visible, j = k1-1 > q0 is not), kt < qt decided by the
// key tile's min and max of se.
//
// Three launches: one block per (row, key tile) reduces se to min/max (reads
// 4*T bytes per row); one block per (row, tile index b) writes row b of the
// class matrix, the compacted list of non-empty key tiles of query tile b
// (ascending, with each key tile's rank in it) and the list of non-empty query
// tiles of key tile b; one block per row numbers the row's non-empty pairs
// (query-tile major) and gives every key-tile list entry its pair index, which
// addresses the backward's per-pair dS tiles.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"
#include "layout.h"

namespace stp {

__global__ void __launch_bounds__(128) tile_minmax_kernel(const int32_t* __restrict__ se, int T,
                                                          int NT, int32_t* __restrict__ kmin,
                                                          int32_t* __restrict__ kmax,
                                                          uint32_t* __restrict__ err) {
  const int kt = blockIdx.x, r = blockIdx.y, t = threadIdx.x;
  const int j = kt * kTile + t;
  int v = se[(size_t)r * T + j];
  if (v < j || v >= T) atomicOr(err, kErrBadSubtreeEnd);
  int mn = v, mx = v;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  __shared__ int smn[4], smx[4];
  if ((t & 31) == 0) {
    smn[t >> 5] = mn;
    smx[t >> 5] = mx;
  }
  __syncthreads();
  if (t == 0) {
    kmin[(size_t)r * NT + kt] = min(min(smn[0], smn[1]), min(smn[2], smn[3]));
    kmax[(size_t)r * NT + kt] = max(max(smx[0], smx[1]), max(smx[2], smx[3]));
  }
}

__device__ __forceinline__ int8_t tile_class(int qt, int kt, int kmn, int kmx) {
  if (kt > qt) return kEmpty;
  if (kt == qt) return kPartial;
  const int q0 = qt * kTile, q1 = q0 + kTile;
  if (kmn >= q1 - 1) return kFull;
  if (kmx < q0) return kEmpty;
  return kPartial;
}

// Exclusive prefix count of `flag` over the 128 threads of the block;
// returns the thread's position and writes the block total to *total.
__device__ __forceinline__ int block_scan128(bool flag, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const unsigned b = __ballot_sync(0xffffffffu, flag);
  if (lane == 0) s_warp[w] = __popc(b);
  __syncthreads();
  int before = 0;
  for (int k = 0; k < w; ++k) before += s_warp[k];
  *total = s_warp[0] + s_warp[1] + s_warp[2] + s_warp[3];
  const int pos = before + __popc(b & ((1u << lane) - 1u));
  __syncthreads();
  return pos;
}

__global__ void __launch_bounds__(128) tile_lists_kernel(int NT, const int32_t* __restrict__ kmin,
                                                         const int32_t* __restrict__ kmax,
                                                         int8_t* __restrict__ cls,
                                                         int32_t* __restrict__ csr_cnt,
                                                         int32_t* __restrict__ csr,
                                                         int32_t* __restrict__ csc_cnt,
                                                         int32_t* __restrict__ csc,
                                                         int32_t* __restrict__ crank) {
  __shared__ int s_warp[4];
  const int b = blockIdx.x, r = blockIdx.y, t = threadIdx.x;
  const int32_t* mn = kmin + (size_t)r * NT;
  const int32_t* mx = kmax + (size_t)r * NT;
  // query tile b: its class row and its key-tile list
  {
    int8_t* crow = cls + ((size_t)r * NT + b) * NT;
    int32_t* list = csr + ((size_t)r * NT + b) * NT;
    int32_t* rank = crank + ((size_t)r * NT + b) * NT;
    int base = 0;
    for (int k0 = 0; k0 < NT; k0 += 128) {
      const int kt = k0 + t;
      int8_t c = kEmpty;
      if (kt < NT) {
        c = tile_class(b, kt, mn[kt], mx[kt]);
        crow[kt] = c;
      }
      int tot;
      const int pos = block_scan128(c != kEmpty, s_warp, &tot);
      if (c != kEmpty) {
        list[base + pos] = (kt << 1) | (c == kPartial ? 1 : 0);
        rank[kt] = base + pos;
      }
      base += tot;
    }
    if (t == 0) csr_cnt[(size_t)r * NT + b] = base;
  }
  // key tile b: its query-tile list
  {
    int32_t* list = csc + ((size_t)r * NT + b) * NT;
    const int kmn = mn[b], kmx = mx[b];
    int base = 0;
    for (int q0 = 0; q0 < NT; q0 += 128) {
      const int qt = q0 + t;
      int8_t c = qt < NT ? tile_class(qt, b, kmn, kmx) : kEmpty;
      int tot;
      const int pos = block_scan128(c != kEmpty, s_warp, &tot);
      if (c != kEmpty) list[base + pos] = (qt << 1) | (c == kPartial ? 1 : 0);
      base += tot;
    }
    if (t == 0) csc_cnt[(size_t)r * NT + b] = base;
  }
}

// One block (1024 threads) per row: exclusive scan of the row's csr counts
// (NT <= 1024) into csr_off, and a contiguous range of pair indices for the
// row taken from a global counter (rows in any order) into row_base.
__global__ void __launch_bounds__(1024) tile_pairs_kernel(int NT, int64_t cap,
                                                          const int32_t* __restrict__ csr_cnt,
                                                          int32_t* __restrict__ csr_off,
                                                          int32_t* __restrict__ row_base,
                                                          int32_t* __restrict__ pair_count,
                                                          uint32_t* __restrict__ err) {
  __shared__ int s_warp[32];
  const int r = blockIdx.x, t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int c = t < NT ? csr_cnt[(size_t)r * NT + t] : 0;
  int x = c;  // inclusive scan: within the warp, then over warp totals
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[w] = x;
  __syncthreads();
  if (w == 0) {
    int v = s_warp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    s_warp[lane] = v;
  }
  __syncthreads();
  const int incl = x + (w > 0 ? s_warp[w - 1] : 0);
  if (t < NT) csr_off[(size_t)r * NT + t] = incl - c;
  if (t == 1023) {
    const int total = incl;
    const int base = atomicAdd(pair_count, total);
    if ((int64_t)base + total > cap) atomicOr(err, kErrCapacity);
    row_base[r] = base;
  }
}

// One block per (key tile, row): the pair index of every entry of the key
// tile's query list, row_base[r] + csr_off[r][qt] + the key tile's rank in
// the query tile's list.
__global__ void __launch_bounds__(128) tile_pair_index_kernel(int NT, const int32_t* __restrict__ csc_cnt,
                                                              const int32_t* __restrict__ csc,
                                                              const int32_t* __restrict__ crank,
                                                              const int32_t* __restrict__ csr_off,
                                                              const int32_t* __restrict__ row_base,
                                                              int32_t* __restrict__ csc_pair) {
  const int kt = blockIdx.x, r = blockIdx.y;
  const int n = csc_cnt[(size_t)r * NT + kt];
  const int base = row_base[r];
  const size_t at = ((size_t)r * NT + kt) * NT;
  for (int e = threadIdx.x; e < n; e += blockDim.x) {
    const int qt = csc[at + e] >> 1;
    csc_pair[at + e] = base + csr_off[(size_t)r * NT + qt] + crank[((size_t)r * NT + qt) * NT + kt];
  }
}

// The launches after min / max: lists, ranks, pair numbering.
cudaError_t launch_lists(const stp_attn_desc* d, const int32_t* kmin, const int32_t* kmax,
                         char* base, const TileMeta& m, uint32_t* err, cudaStream_t s) {
  const int NT = d->row_len / kTile;
  dim3 grid(NT, d->n_rows);
  int32_t* pair_count = reinterpret_cast<int32_t*>(base + m.pair_count);
  cudaError_t e = cudaMemsetAsync(pair_count, 0, 4, s);
  if (e != cudaSuccess) return e;
  tile_lists_kernel<<<grid, 128, 0, s>>>(
      NT, kmin, kmax, reinterpret_cast<int8_t*>(base + m.cls),
      reinterpret_cast<int32_t*>(base + m.csr_cnt), reinterpret_cast<int32_t*>(base + m.csr),
      reinterpret_cast<int32_t*>(base + m.csc_cnt), reinterpret_cast<int32_t*>(base + m.csc),
      reinterpret_cast<int32_t*>(base + m.crank));
  tile_pairs_kernel<<<d->n_rows, 1024, 0, s>>>(
      NT, pair_capacity(d->n_rows, NT, d->max_tile_pairs), reinterpret_cast<const int32_t*>(base + m.csr_cnt),
      reinterpret_cast<int32_t*>(base + m.csr_off), reinterpret_cast<int32_t*>(base + m.row_base), pair_count, err);
  tile_pair_index_kernel<<<grid, 128, 0, s>>>(
      NT, reinterpret_cast<const int32_t*>(base + m.csc_cnt), reinterpret_cast<const int32_t*>(base + m.csc),
      reinterpret_cast<const int32_t*>(base + m.crank), reinterpret_cast<const int32_t*>(base + m.csr_off),
      reinterpret_cast<const int32_t*>(base + m.row_base), reinterpret_cast<int32_t*>(base + m.csc_pair));
  return cudaGetLastError();
}

}  // namespace stp

using namespace stp;

extern "C" stp_status stp_count_tile_pairs(const int32_t* subtree_end, int32_t n_rows,
                                           int32_t row_len, int64_t* n_pairs) {
  clear_error();
  if (!n_pairs || (!subtree_end && n_rows > 0)) return fail(STP_EINVAL, "stp_count_tile_pairs: NULL pointer");
  if (n_rows < 0 || row_len <= 0 || row_len % kTile)
    return fail(STP_EINVAL, "stp_count_tile_pairs: need n_rows >= 0 and row_len a positive multiple of 128");
  int64_t total = 0;
  for (int64_t r = 0; r < n_rows; ++r) {
    const int32_t* se = subtree_end + r * row_len;
    for (int32_t k0 = 0; k0 < row_len; k0 += kTile) {
      int32_t mx = -1;
      for (int32_t j = k0; j < k0 + kTile; ++j) {
        if (se[j] < j || se[j] >= row_len)
          return fail(STP_EINVAL, "stp_count_tile_pairs: subtree_end[%lld][%d] = %d outside [j, row_len)",
                      (long long)r, j, se[j]);
        mx = se[j] > mx ? se[j] : mx;
      }
      total += mx / kTile - k0 / kTile + 1;
    }
  }
  *n_pairs = total;
  return STP_OK;
}


extern "C" stp_status stp_workspace_size(const stp_attn_desc* desc, size_t* tile_meta_bytes,
                                         size_t* fwd_ws_bytes, size_t* bwd_ws_bytes) {
  clear_error();
  stp_status st = check_desc(desc);
  if (st) return st;
  const int64_t NT = desc->row_len / kTile;
  if (tile_meta_bytes) *tile_meta_bytes = tile_meta_layout(desc->n_rows, NT).total;
  if (fwd_ws_bytes) *fwd_ws_bytes = 256;
  if (bwd_ws_bytes)
    *bwd_ws_bytes = bwd_ws_layout(desc->n_rows, desc->row_len, desc->n_q_heads, desc->n_kv_heads,
                                  desc->dtype == STP_BF16, pair_capacity(desc->n_rows, NT, desc->max_tile_pairs),
                                  desc->ds_groups)
                        .total;
  return STP_OK;
}

extern "C" stp_status stp_classify(const stp_attn_desc* desc, const int32_t* d_subtree_end,
                                   void* d_tile_meta, void* stream) {
  clear_error();
  stp_status st = check_desc(desc);
  if (st) return st;
  if (!d_subtree_end || !d_tile_meta) return fail(STP_EINVAL, "stp_classify: NULL device pointer");
  if ((reinterpret_cast<uintptr_t>(d_tile_meta) & 255) || (reinterpret_cast<uintptr_t>(d_subtree_end) & 15))
    return fail(STP_EINVAL, "stp_classify: tile_meta must be 256-byte and subtree_end 16-byte aligned");
  if (desc->n_rows == 0) return STP_OK;
  const int NT = desc->row_len / kTile;
  const TileMeta m = tile_meta_layout(desc->n_rows, NT);
  char* base = static_cast<char*>(d_tile_meta);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t* err = reinterpret_cast<uint32_t*>(base + m.err);
  cudaMemsetAsync(err, 0, 4, s);
  dim3 grid(NT, desc->n_rows);
  tile_minmax_kernel<<<grid, 128, 0, s>>>(d_subtree_end, desc->row_len, NT,
                                          reinterpret_cast<int32_t*>(base + m.kmin),
                                          reinterpret_cast<int32_t*>(base + m.kmax), err);
  cudaError_t e = launch_lists(desc, reinterpret_cast<const int32_t*>(base + m.kmin),
                               reinterpret_cast<const int32_t*>(base + m.kmax), base, m, err, s);
  if (e != cudaSuccess) return fail(STP_ECUDA, "stp_classify: %s", cudaGetErrorString(e));
  return STP_OK;
}

extern "C" stp_status stp_read_tile_classes(const stp_attn_desc* desc, const void* d_tile_meta,
                                            int8_t* d_cls_out, void* stream) {
  clear_error();
  stp_status st = check_desc(desc);
  if (st) return st;
  if (!d_tile_meta || !d_cls_out) return fail(STP_EINVAL, "stp_read_tile_classes: NULL pointer");
  const int64_t NT = desc->row_len / kTile;
  const TileMeta m = tile_meta_layout(desc->n_rows, NT);
  const size_t n = size_t(desc->n_rows) * NT * NT;
  if (n == 0) return STP_OK;
  cudaError_t e = cudaMemcpyAsync(d_cls_out, static_cast<const char*>(d_tile_meta) + m.cls, n,
                                  cudaMemcpyDeviceToDevice, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(STP_ECUDA, "stp_read_tile_classes: %s", cudaGetErrorString(e));
  return STP_OK;
}

extern "C" stp_status stp_device_status(const void* d_ws, void* stream, stp_status* out) {
  clear_error();
  if (!d_ws || !out) return fail(STP_EINVAL, "stp_device_status: NULL pointer");
  uint32_t word = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(&word, d_ws, 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail(STP_ECUDA, "stp_device_status: %s", cudaGetErrorString(e));
  *out = word ? STP_EDEVICE : STP_OK;
  if (word) fail(STP_EDEVICE, "device error word 0x%x", word);
  return STP_OK;
}

// ---------------------------------------------------------------------------
// Classification for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where
// they classify: code recording a CUDA graph, a plug-in host that only hands
// over the buffers of its inputs and outputs, or a latency-critical loop that
// forbids allocation.  This variant keeps its only scratch -- the per-key-tile
// min / max of subtree_end -- in a fixed array owned by the library instead
// of in the caller's buffer.  The array is a file-scope device variable: every
// GPU that loads the library holds it (1 MiB) until the process exits.
// ---------------------------------------------------------------------------

constexpr int64_t kNoAllocMaxTiles = 131072;  // rows x (row_len / 128), at most
static __device__ __align__(256) int32_t g_classify_scratch[2 * kNoAllocMaxTiles];

namespace {

constexpr int kMaxDevices = 64;

// Device address of g_classify_scratch on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device, with that device current, and cached.
stp_status classify_scratch(int32_t** out) {
  static std::mutex mu;
  static int32_t* addr[kMaxDevices] = {};
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(STP_ECUDA, "stp_classify_noalloc: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(STP_EUNSUPPORTED, "device ordinal %d >= %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_classify_scratch);
    if (e != cudaSuccess || !p)
      return fail(STP_ECUDA, "stp_classify_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    addr[dev] = static_cast<int32_t*>(p);
  }
  *out = addr[dev];
  return STP_OK;
}

}  // namespace

extern "C" stp_status stp_classify_noalloc(const stp_attn_desc* desc, const int32_t* d_subtree_end,
                                           void* d_tile_meta, void* stream) {
  clear_error();
  stp_status st = check_desc(desc);
  if (st) return st;
  if (!d_subtree_end || !d_tile_meta)
    return fail(STP_EINVAL, "stp_classify_noalloc: NULL device pointer");
  if ((reinterpret_cast<uintptr_t>(d_tile_meta) & 255) || (reinterpret_cast<uintptr_t>(d_subtree_end) & 15))
    return fail(STP_EINVAL, "stp_classify_noalloc: tile_meta must be 256-byte and subtree_end 16-byte aligned");
  const int64_t NT = desc->row_len / kTile;
  if ((int64_t)desc->n_rows * NT > kNoAllocMaxTiles)
    return fail(STP_EINVAL,
                "stp_classify_noalloc: %d rows x %lld tiles exceed the fixed scratch of %lld tiles "
                "(use stp_classify)",
                desc->n_rows, (long long)NT, (long long)kNoAllocMaxTiles);
  if (desc->n_rows == 0) return STP_OK;
  int32_t* scratch = nullptr;
  st = classify_scratch(&scratch);
  if (st) return st;
  const TileMeta m = tile_meta_layout(desc->n_rows, NT);
  char* base = static_cast<char*>(d_tile_meta);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t* err = reinterpret_cast<uint32_t*>(base + m.err);
  cudaMemsetAsync(err, 0, 4, s);
  // every min / max entry is written before it is read: nothing to clear
  int32_t* kmin = scratch;
  int32_t* kmax = scratch + kNoAllocMaxTiles;
  dim3 grid((unsigned)NT, desc->n_rows);
  tile_minmax_kernel<<<grid, 128, 0, s>>>(d_subtree_end, desc->row_len, (int)NT, kmin, kmax, err);
  cudaError_t e = launch_lists(desc, kmin, kmax, base, m, err, s);
  if (e != cudaSuccess) return fail(STP_ECUDA, "stp_classify_noalloc: %s", cudaGetErrorString(e));
  return STP_OK;
}
