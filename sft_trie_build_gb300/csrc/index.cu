// Tree-aware top-k indexer ("Prefix tree packing", attention section, the
// sparse top-k indexer variants): sparse attention gathers the key indices it
// is handed, so the tree lives in the indexer, which scores candidates from a
// query's own ancestor chain only (the enter/exit interval check of the mask)
// and never proposes a sibling branch's keys.
//
//   score(i, j) = sum_h w[i, h] * max(q[i, h] . k[j], 0)   for visible j
//   top-k(i)    = the k visible keys of largest score, ties to the smaller
//                 key index, listed in ascending key order (padded with -1).
//
// Two kernels, both driven by the per-query-tile key-tile lists and the pair
// numbering of stp_classify:
//   index_scores_kernel  one CTA per (row, query tile, piece of at most 8
//                        entries of its key-tile list, so long ancestor lists
//                        spread over the chip): the tile's Q of every
//                        indexer head once (TMA), the piece's key tiles
//                        through a two-stage ring; S_h = Q_h K^T on tcgen05
//                        (four heads per pass in TMEM), and four epilogue
//                        warps (thread = query = TMEM lane) accumulate
//                        w * relu(S) in registers, apply the predicate on
//                        PARTIAL tiles and write the tile's scores key-major
//                        ([128 keys][128 queries] fp32) to the pair's slot.
//   index_select_kernel  one CTA per (row, query tile): byte-wise radix
//                        select of each query's k-th largest candidate score
//                        (histograms in shared memory), then the keys above
//                        it, and the ties it needs, emitted in ascending order.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"
#include "layout.h"
#include "tc_ptx.cuh"

namespace stp {
namespace {

using namespace tc;

constexpr int kIdxThreads = 192;       // warps 0-3 epilogue, warp 4 TMA, warp 5 MMA
constexpr int kIdxSlots = 4;           // heads per TMEM pass (128 columns each)
constexpr int kIdxQBytesMax = 131072;  // Q of all heads: H * D * 256 bytes
constexpr int kIdxSmallBytes = 256;
constexpr int kScoreTile = 128 * 128;  // floats per (pair) score tile
constexpr int kIdxPiece = 8;           // key tiles of one query tile's list per scoring CTA
constexpr int kSelThreads = 1024;  // 32 warps: 2 query groups x 16 key-tile ranges
constexpr int kSelQ = 64;          // queries per selection CTA (half a query tile)
constexpr int kSelSplit = 32 / (kSelQ / 32);

struct IdxParams {
  int R, T, NT, H, D, top_k, splits;   // splits: scoring CTAs per query tile
  int64_t cap;
  const int32_t* se;
  const int32_t* csr_cnt;
  const int32_t* csr;
  const int32_t* csr_off;
  const int32_t* row_base;
  const float* w;       // [R*T, H]
  float* scores;        // [cap][128 keys][128 queries]
  int32_t* out_idx;     // [R*T, k]
  float* out_score;     // [R*T, k]
  uint32_t* err;
};

enum { X_Q = 0, X_KF = 1, X_KE = 3, X_SF = 5, X_SFREE = 6, X_DRAIN = 7, X_COUNT = 8 };

typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                             const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                             CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  });
  return fn;
}

// [rows, H, D] bf16 as a 3-D tensor (d, head, row); 64 d x 1 head x 128 rows
// boxes, 128-byte swizzled.
bool make_map_d(CUtensorMap* m, const void* base, int64_t rows, int H, int D) {
  EncodeFn enc = encode();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
  cuuint32_t box[3] = {64, 1, 128};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

__global__ void __launch_bounds__(kIdxThreads, 1)
    index_scores_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                        const IdxParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int tile_bytes = 128 * p.D * 2;          // one 128-row tile of one head
  const int q_bytes = p.H * tile_bytes;
  uint8_t* big = smem_raw;
  const uint32_t big_s = smem_u32(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw + q_bytes + 2 * tile_bytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + X_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CTA = (query tile, piece of at most kIdxPiece entries of its key-tile list)
  const int piece = (int)(blockIdx.x % p.splits), rest = (int)(blockIdx.x / p.splits);
  const int qt = p.NT - 1 - rest / p.R;   // longest lists first
  const int r = rest % p.R;
  const int cnt = p.csr_cnt[(size_t)r * p.NT + qt];
  const int e0 = piece * kIdxPiece, e1 = cnt < e0 + kIdxPiece ? cnt : e0 + kIdxPiece;
  if (piece > 0 && e0 >= cnt) return;   // uniform over the CTA; piece 0 always checks the list
  const int32_t* list = p.csr + ((size_t)r * p.NT + qt) * p.NT;
  const int64_t pbase = (int64_t)p.row_base[r] + p.csr_off[(size_t)r * p.NT + qt];
  const int row0 = r * p.T;
  const int n_groups = (p.H + kIdxSlots - 1) / kIdxSlots;

  if (threadIdx.x == 0) {
    for (int b = 0; b < X_COUNT; ++b) mbar_init(&bars[b], b == X_SFREE ? 4 : 1);
    *abort_flag = 0;
    if ((big_s & 1023u) != 0 || cnt <= 0 || cnt > p.NT) {
      *abort_flag = 1;
      atomicOr(p.err, (big_s & 1023u) != 0 ? kErrTmem : kErrBadList);
    }
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const bool run = !*abort_flag;

  if (warp == 4) {
    if (lane == 0 && run) {
      // ------------------------------------------------------------ loads
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      mbar_expect_tx(&bars[X_Q], (uint32_t)q_bytes);
      for (int h = 0; h < p.H; ++h)
        for (int db = 0; db < p.D / 64; ++db)
          tma_load_3d(big + h * tile_bytes + db * 16384, &tq, &bars[X_Q], db * 64, h, row0 + qt * 128);
      int issued[2] = {-1, -1};
      for (int e = e0; e < e1; ++e) {
        const int st = (e - e0) & 1, n = (e - e0) >> 1, kt = list[e] >> 1;
        if (kt < 0 || kt > qt) {
          *abort_flag = 1;
          atomicOr(p.err, kErrBadList);
          break;
        }
        if (e >= 2 && !mbar_wait(&bars[X_KE + st], (n - 1) & 1, abort_flag, p.err)) break;
        mbar_expect_tx(&bars[X_KF + st], (uint32_t)tile_bytes);
        for (int db = 0; db < p.D / 64; ++db)
          tma_load_3d(big + q_bytes + st * tile_bytes + db * 16384, &tk, &bars[X_KF + st], db * 64, 0,
                      row0 + kt * 128);
        issued[st] = n;
      }
      mbar_wait_drain(&bars[X_Q], 0);
      for (int st = 0; st < 2; ++st)
        if (issued[st] >= 0) mbar_wait_drain(&bars[X_KF + st], issued[st] & 1);
    }
    __syncwarp();
  } else if (warp == 5) {
    if (lane == 0 && run) {
      // ------------------------------------------------------------ MMA
      constexpr uint32_t idesc = idesc_bf16(128, 128, 0, 0);
      auto km = [](int kk) { return (uint32_t)((kk >> 2) * (16384 >> 4) + (kk & 3) * 2); };
      const int nk = p.D / 16;
      bool ok = mbar_wait(&bars[X_Q], 0, abort_flag, p.err);
      int u = 0;  // head passes issued so far
      for (int e = e0; ok && e < e1; ++e) {
        const int st = (e - e0) & 1;
        if (!mbar_wait(&bars[X_KF + st], ((e - e0) >> 1) & 1, abort_flag, p.err)) break;
        const uint32_t k_km = desc_lo_kmajor(big_s + q_bytes + st * tile_bytes);
        for (int hg = 0; ok && hg < n_groups; ++hg, ++u) {
          if (u > 0 && !mbar_wait(&bars[X_SFREE], (u - 1) & 1, abort_flag, p.err)) {
            ok = false;
            break;
          }
          fence_after_sync();
          for (int hs = 0; hs < kIdxSlots && kIdxSlots * hg + hs < p.H; ++hs) {
            const uint32_t q_km = desc_lo_kmajor(big_s + (kIdxSlots * hg + hs) * tile_bytes);
            for (int kk = 0; kk < nk; ++kk) mma_ss_lo(tmem + hs * 128, q_km + km(kk), k_km + km(kk), idesc, kk > 0);
          }
          mma_commit(&bars[X_SF]);
        }
        if (ok) mma_commit(&bars[X_KE + st]);
      }
      mma_commit(&bars[X_DRAIN]);
      mbar_wait_drain(&bars[X_DRAIN], 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int il = threadIdx.x;                 // query row = TMEM lane
    const int i = qt * 128 + il;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float* wrow = p.w + ((size_t)row0 + i) * p.H;
    bool ok = run;
    int u = 0;
    for (int e = e0; ok && e < e1; ++e) {
      const int ent = list[e], kt = ent >> 1, part = ent & 1;
      float acc[128];
#pragma unroll
      for (int j = 0; j < 128; ++j) acc[j] = 0.f;
      for (int hg = 0; hg < n_groups; ++hg, ++u) {
        if (!__all_sync(0xffffffffu, mbar_wait(&bars[X_SF], u & 1, abort_flag, p.err))) {
          ok = false;
          break;
        }
        fence_after_sync();
        for (int hs = 0; hs < kIdxSlots && kIdxSlots * hg + hs < p.H; ++hs) {
          const float wi = wrow[kIdxSlots * hg + hs];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t x[32];
            tmem_ld32(tmem + lane_base + hs * 128 + c * 32, x);
            tmem_ld_wait();
#pragma unroll
            for (int m = 0; m < 32; ++m) acc[c * 32 + m] = fmaf(wi, fmaxf(__uint_as_float(x[m]), 0.f), acc[c * 32 + m]);
          }
        }
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[X_SFREE]);
      }
      if (!ok) break;
      const int64_t pair = pbase + e;
      if (pair < 0 || pair >= p.cap) {
        atomicOr(p.err, kErrCapacity);
        continue;
      }
      float* out = p.scores + (size_t)pair * kScoreTile + il;
      const int32_t* se_tile = p.se + (size_t)row0 + kt * 128;
#pragma unroll
      for (int j = 0; j < 128; ++j) {
        const int jk = kt * 128 + j;
        const bool vis = !part || (jk <= i && __ldg(se_tile + j) >= i);
        out[j * 128] = vis ? acc[j] : -INFINITY;   // key-major: a warp writes 128 contiguous bytes
      }
    }
  }

  __syncwarp();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == 5) tmem_dealloc(tmem, 512);
}

// float -> uint32 with the same order (larger float, larger key)
__device__ __forceinline__ uint32_t order_key(float s) {
  const uint32_t u = __float_as_uint(s);
  return (u >> 31) ? ~u : (u | 0x80000000u);
}

// One CTA per (row, half a query tile), 32 warps: warp w serves queries
// 32 (w % 2) .. +31 of the half (lane = query) over the (w / 2)-th of sixteen
// contiguous ranges of the tile's key-tile list.  Four byte-wise radix passes build each
// query's histogram in shared memory (atomics across the eight ranges) and
// pin the k-th largest score; a counting pass then gives every range its
// output offset, so the ranges emit in parallel and the keys still come out
// in ascending order, ties to the smaller key index.
__global__ void __launch_bounds__(kSelThreads) index_select_kernel(const IdxParams p) {
  extern __shared__ uint32_t hist[];   // [256 bins][kSelQ queries]
  __shared__ uint32_t s_prefix[kSelQ], s_mask[kSelQ];
  __shared__ int s_rem[kSelQ], s_all[kSelQ];
  __shared__ int s_gt[kSelSplit][kSelQ], s_eq[kSelSplit][kSelQ];
  constexpr int kHalves = 128 / kSelQ;
  const int qt = p.NT - 1 - (int)(blockIdx.x / (p.R * kHalves));
  const int r = (int)(blockIdx.x / kHalves % p.R), half = (int)(blockIdx.x % kHalves);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kGroups = kSelQ / 32;
  const int qg = warp % kGroups, ts = warp / kGroups;
  const int ql = qg * 32 + lane;               // query within the CTA
  const int il = half * kSelQ + ql, i = qt * 128 + il;
  const int cnt = p.csr_cnt[(size_t)r * p.NT + qt];
  const int32_t* list = p.csr + ((size_t)r * p.NT + qt) * p.NT;
  const int64_t pbase = (int64_t)p.row_base[r] + p.csr_off[(size_t)r * p.NT + qt];
  const int k = p.top_k;
  int32_t* oi = p.out_idx + ((size_t)r * p.T + i) * k;
  float* os = p.out_score + ((size_t)r * p.T + i) * k;
  if (cnt <= 0 || cnt > p.NT || pbase + cnt > p.cap) {   // uniform over the CTA
    if (threadIdx.x == 0) atomicOr(p.err, cnt <= 0 || cnt > p.NT ? kErrBadList : kErrCapacity);
    if (ts == 0)
      for (int n = 0; n < k; ++n) {
        oi[n] = -1;
        os[n] = -INFINITY;
      }
    return;
  }
  const int e0 = ts * cnt / kSelSplit, e1 = (ts + 1) * cnt / kSelSplit;
  auto tile = [&](int e) { return p.scores + (size_t)(pbase + e) * kScoreTile + il; };
  if (threadIdx.x < kSelQ) {
    s_prefix[threadIdx.x] = 0;
    s_mask[threadIdx.x] = 0;
    s_rem[threadIdx.x] = k;
    s_all[threadIdx.x] = 0;
  }
  for (int b = 3; b >= 0; --b) {
    for (int x = threadIdx.x; x < 256 * kSelQ; x += kSelThreads) hist[x] = 0;
    __syncthreads();
    const uint32_t prefix = s_prefix[ql], mask = s_mask[ql];
    if (!s_all[ql]) {
      for (int e = e0; e < e1; ++e) {
        const float* t = tile(e);
        for (int j = 0; j < 128; ++j) {
          const float sc = t[j * 128];
          if (sc == -INFINITY) continue;
          const uint32_t key = order_key(sc);
          if ((key & mask) == prefix) atomicAdd(&hist[((key >> (8 * b)) & 255u) * kSelQ + ql], 1u);
        }
      }
    }
    __syncthreads();
    if (threadIdx.x < kSelQ) {
      const int q = threadIdx.x;
      if (b == 3) {
        int total = 0;
        for (int bin = 0; bin < 256; ++bin) total += (int)hist[bin * kSelQ + q];
        if (total <= k) s_all[q] = 1;
      }
      if (!s_all[q]) {
        const int remaining = s_rem[q];
        int cum = 0;
        for (int bin = 255; bin >= 0; --bin) {
          const int c = (int)hist[bin * kSelQ + q];
          if (cum + c >= remaining) {
            s_prefix[q] |= (uint32_t)bin << (8 * b);
            s_rem[q] = remaining - cum;
            break;
          }
          cum += c;
        }
        s_mask[q] |= 255u << (8 * b);
      }
    }
    __syncthreads();
  }
  const uint32_t thr = s_prefix[ql];
  const int ties = s_rem[ql];
  const bool all = s_all[ql] != 0;
  // counting pass: keys above the threshold and keys equal to it, per range
  int gt = 0, eq = 0;
  for (int e = e0; e < e1; ++e) {
    const float* t = tile(e);
    for (int j = 0; j < 128; ++j) {
      const float sc = t[j * 128];
      if (sc == -INFINITY) continue;
      if (all) {
        ++gt;
      } else {
        const uint32_t key = order_key(sc);
        gt += key > thr;
        eq += key == thr;
      }
    }
  }
  s_gt[ts][ql] = gt;
  s_eq[ts][ql] = eq;
  __syncthreads();
  int before = 0, eq_before = 0;
  for (int t2 = 0; t2 < ts; ++t2) {
    before += s_gt[t2][ql];
    eq_before += s_eq[t2][ql];
  }
  int n = before + (all ? 0 : min(ties, eq_before));
  int my_ties = all ? 0 : max(0, min(eq, ties - eq_before));
  for (int e = e0; e < e1; ++e) {
    const float* t = tile(e);
    const int kt = list[e] >> 1;
    for (int j = 0; j < 128; ++j) {
      const float sc = t[j * 128];
      if (sc == -INFINITY) continue;
      bool take = all;
      if (!all) {
        const uint32_t key = order_key(sc);
        take = key > thr || (key == thr && my_ties > 0);
        if (key == thr && my_ties > 0) --my_ties;
      }
      if (take) {
        oi[n] = kt * 128 + j;
        os[n] = sc;
        ++n;
      }
    }
  }
  if (ts == kSelSplit - 1)
    for (; n < k; ++n) {
      oi[n] = -1;
      os[n] = -INFINITY;
    }
}

stp_status check_index_desc(const stp_index_desc* d) {
  if (!d) return fail(STP_EINVAL, "index descriptor is NULL");
  if (d->n_rows < 0) return fail(STP_EINVAL, "n_rows < 0");
  if (d->row_len <= 0 || d->row_len % kTile || d->row_len > kMaxRowLen)
    return fail(STP_EUNSUPPORTED, "row_len %d must be a positive multiple of 128 and <= %d", d->row_len, kMaxRowLen);
  if (d->head_dim != 64 && d->head_dim != 128) return fail(STP_EUNSUPPORTED, "head_dim must be 64 or 128");
  if (d->n_heads < 1 || (int64_t)d->n_heads * d->head_dim * 256 > kIdxQBytesMax)
    return fail(STP_EUNSUPPORTED, "need n_heads >= 1 and n_heads * head_dim <= 512 (got %d x %d)", d->n_heads,
                d->head_dim);
  if (d->top_k < 1 || d->top_k > 4096) return fail(STP_EUNSUPPORTED, "top_k must lie in [1, 4096]");
  if (d->max_tile_pairs < 0) return fail(STP_EINVAL, "max_tile_pairs must be >= 0");
  return STP_OK;
}

}  // namespace
}  // namespace stp

using namespace stp;

extern "C" stp_status stp_index_workspace_size(const stp_index_desc* desc, size_t* ws_bytes) {
  clear_error();
  stp_status st = check_index_desc(desc);
  if (st) return st;
  if (!ws_bytes) return fail(STP_EINVAL, "stp_index_workspace_size: NULL output");
  const int64_t cap = pair_capacity(desc->n_rows, desc->row_len / kTile, desc->max_tile_pairs);
  *ws_bytes = 256 + (size_t)cap * kScoreTile * sizeof(float);
  return STP_OK;
}

extern "C" stp_status stp_index_topk(const stp_index_desc* desc, const void* q, const void* k,
                                     const float* w, const int32_t* d_subtree_end,
                                     const void* d_tile_meta, int32_t* topk_idx, float* topk_score,
                                     void* d_ws, void* stream) {
  clear_error();
  stp_status st = check_index_desc(desc);
  if (st) return st;
  if (!q || !k || !w || !d_subtree_end || !d_tile_meta || !topk_idx || !topk_score || !d_ws)
    return fail(STP_EINVAL, "stp_index_topk: NULL device pointer");
  auto mis = [](const void* x, uintptr_t a) { return (reinterpret_cast<uintptr_t>(x) & (a - 1)) != 0; };
  if (mis(q, 16) || mis(k, 16) || mis(w, 4) || mis(d_tile_meta, 256) || mis(d_ws, 256))
    return fail(STP_EINVAL, "stp_index_topk: q, k 16-byte, tile_meta and ws 256-byte aligned");
  if (desc->n_rows == 0) return STP_OK;
  const int NT = desc->row_len / kTile;
  const TileMeta m = tile_meta_layout(desc->n_rows, NT);
  const char* tm = static_cast<const char*>(d_tile_meta);
  IdxParams p;
  p.R = desc->n_rows;
  p.T = desc->row_len;
  p.NT = NT;
  p.H = desc->n_heads;
  p.D = desc->head_dim;
  p.top_k = desc->top_k;
  p.cap = pair_capacity(desc->n_rows, NT, desc->max_tile_pairs);
  p.se = d_subtree_end;
  p.csr_cnt = reinterpret_cast<const int32_t*>(tm + m.csr_cnt);
  p.csr = reinterpret_cast<const int32_t*>(tm + m.csr);
  p.csr_off = reinterpret_cast<const int32_t*>(tm + m.csr_off);
  p.row_base = reinterpret_cast<const int32_t*>(tm + m.row_base);
  p.w = w;
  p.err = static_cast<uint32_t*>(d_ws);
  p.scores = reinterpret_cast<float*>(static_cast<char*>(d_ws) + 256);
  p.out_idx = topk_idx;
  p.out_score = topk_score;
  const int64_t rows = (int64_t)desc->n_rows * desc->row_len;
  CUtensorMap mq, mk;
  if (!make_map_d(&mq, q, rows, p.H, p.D) || !make_map_d(&mk, k, rows, 1, p.D))
    return fail(STP_ECUDA, "stp_index_topk: tensor map encoding failed");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(p.err, 0, 4, s);
  const int smem = p.H * 128 * p.D * 2 + 2 * 128 * p.D * 2 + kIdxSmallBytes;
  const int smem_sel = 256 * kSelQ * 4;
  static bool attr = false;
  if (e == cudaSuccess && !attr) {
    e = cudaFuncSetAttribute(index_scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kIdxQBytesMax + 2 * 128 * 128 * 2 + kIdxSmallBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(index_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_sel);
    attr = e == cudaSuccess;
  }
  if (e != cudaSuccess) return fail(STP_ECUDA, "stp_index_topk: %s", cudaGetErrorString(e));
  const unsigned grid = (unsigned)(NT * desc->n_rows);
  p.splits = (NT + kIdxPiece - 1) / kIdxPiece;
  index_scores_kernel<<<grid * p.splits, kIdxThreads, smem, s>>>(mq, mk, p);
  index_select_kernel<<<grid * (128 / kSelQ), kSelThreads, smem_sel, s>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(STP_ECUDA, "stp_index_topk: %s", cudaGetErrorString(e));
  return STP_OK;
}
