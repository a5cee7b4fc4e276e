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
//                        (two heads per pass, two passes' accumulators in
//                        TMEM, so the next pass runs while the epilogue reads
//                        this one), and eight epilogue
//                        warps (thread = query = TMEM lane, each warp half
//                        of the keys) accumulate
//                        w * relu(S) in registers, apply the predicate on
//                        PARTIAL tiles and write the tile's scores
//                        query-major ([128 queries][128 keys] fp32: one
//                        512-byte row per query) to the pair's slot.
//   index_select_kernel  one warp per query: byte-wise radix select of its
//                        k-th largest candidate score over its score rows (a
//                        256-bin histogram in shared memory per warp),
//                        then the keys above it, and the ties it needs,
//                        emitted in ascending order.
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

constexpr int kIdxThreads = 320;       // warps 0-7 epilogue, warp 8 TMA, warp 9 MMA
constexpr int kIdxTma = 8, kIdxMma = 9;
constexpr int kIdxMaxHeads = 8;        // n_heads * head_dim <= 512 and head_dim >= 64
constexpr int kIdxSlots = 2;           // heads per TMEM pass (128 columns each); two passes' buffers
constexpr int kIdxQBytesMax = 131072;  // Q of all heads: H * D * 256 bytes
constexpr int kIdxSmallBytes = 256;
constexpr int kScoreTile = 128 * 128;  // keys per (pair) score tile
constexpr int kIdxPiece = 8;           // key tiles of one query tile's list per scoring CTA

struct IdxParams {
  int R, T, NT, H, D, top_k, splits;   // splits: scoring CTAs per query tile
  int64_t cap;
  const int32_t* se;
  const int32_t* csr_cnt;
  const int32_t* csr;
  const int32_t* csr_off;
  const int32_t* row_base;
  const float* w;       // [R*T, H]
  uint32_t* scores;     // [cap][128 queries][128 keys]: order keys of the scores, 0 = not visible
  int32_t* out_idx;     // [R*T, k]
  float* out_score;     // [R*T, k]
  uint32_t* err;
};

enum { X_Q = 0, X_KF = 1, X_KE = 3, X_SF = 5, X_SFREE = 7, X_DRAIN = 9, X_COUNT = 10 };

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

// float -> uint32 with the same order (larger float, larger key).  Every
// float but a NaN maps above 0 (-inf to 0x007fffff), so 0 is free to mark a
// key that is not visible.
__device__ __forceinline__ uint32_t order_key(float s) {
  const uint32_t u = __float_as_uint(s);
  return (u >> 31) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t key) {
  return __uint_as_float((key >> 31) ? (key & 0x7fffffffu) : ~key);
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
    for (int b = 0; b < X_COUNT; ++b) mbar_init(&bars[b], (b == X_SFREE || b == X_SFREE + 1) ? 8 : 1);
    *abort_flag = 0;
    if ((big_s & 1023u) != 0 || cnt <= 0 || cnt > p.NT) {
      *abort_flag = 1;
      atomicOr(p.err, (big_s & 1023u) != 0 ? kErrTmem : kErrBadList);
    }
    fence_mbar_init();
  }
  if (warp == kIdxMma) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const bool run = !*abort_flag;

  if (warp == kIdxTma) {
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
  } else if (warp == kIdxMma) {
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
          // pass u fills buffer u & 1 once the epilogue has read pass u - 2 from it
          const int bu = u & 1;
          if (u > 1 && !mbar_wait(&bars[X_SFREE + bu], ((u - 2) >> 1) & 1, abort_flag, p.err)) {
            ok = false;
            break;
          }
          fence_after_sync();
          for (int hs = 0; hs < kIdxSlots && kIdxSlots * hg + hs < p.H; ++hs) {
            const uint32_t q_km = desc_lo_kmajor(big_s + (kIdxSlots * hg + hs) * tile_bytes);
            for (int kk = 0; kk < nk; ++kk)
              mma_ss_lo(tmem + bu * 256 + hs * 128, q_km + km(kk), k_km + km(kk), idesc, kk > 0);
          }
          mma_commit(&bars[X_SF + bu]);
        }
        if (ok) mma_commit(&bars[X_KE + st]);
      }
      mma_commit(&bars[X_DRAIN]);
      mbar_wait_drain(&bars[X_DRAIN], 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // warp w: query rows 32 (w % 4) .. + 31 (thread = TMEM lane), keys 64 (w / 4) .. + 63
    const int il = 32 * (warp & 3) + lane, kh = 64 * (warp >> 2);
    const int i = qt * 128 + il;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    float wreg[kIdxMaxHeads];   // this query's head weights
    {
      const float* wrow = p.w + ((size_t)row0 + i) * p.H;
#pragma unroll
      for (int h = 0; h < kIdxMaxHeads; ++h) wreg[h] = h < p.H ? wrow[h] : 0.f;
    }
    bool ok = run;
    int u = 0;
    for (int e = e0; ok && e < e1; ++e) {
      const int ent = list[e], kt = ent >> 1, part = ent & 1;
      float acc[64];
#pragma unroll
      for (int j = 0; j < 64; ++j) acc[j] = 0.f;
      for (int hg = 0; hg < n_groups; ++hg, ++u) {
        const int bu = u & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&bars[X_SF + bu], (u >> 1) & 1, abort_flag, p.err))) {
          ok = false;
          break;
        }
        fence_after_sync();
#pragma unroll
        for (int hs = 0; hs < kIdxSlots; ++hs) {
          if (kIdxSlots * hg + hs >= p.H) break;
          float wi = wreg[0];
#pragma unroll
          for (int h = 1; h < kIdxMaxHeads; ++h)
            if (h == kIdxSlots * hg + hs) wi = wreg[h];
          uint32_t x[64];
          tmem_ld32(tmem + lane_base + bu * 256 + hs * 128 + kh, x);
          tmem_ld32(tmem + lane_base + bu * 256 + hs * 128 + kh + 32, x + 32);
          tmem_ld_wait();
          const float2 w2 = make_float2(wi, wi);
#pragma unroll
          for (int m = 0; m < 64; m += 2) {   // two columns per packed FFMA
            const float2 r2 = make_float2(fmaxf(__uint_as_float(x[m]), 0.f), fmaxf(__uint_as_float(x[m + 1]), 0.f));
            const float2 a2 = __ffma2_rn(w2, r2, make_float2(acc[m], acc[m + 1]));
            acc[m] = a2.x;
            acc[m + 1] = a2.y;
          }
        }
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[X_SFREE + bu]);
      }
      if (!ok) break;
      const int64_t pair = pbase + e;
      if (pair < 0 || pair >= p.cap) {
        atomicOr(p.err, kErrCapacity);
        continue;
      }
      // query-major: the thread's 64 keys are one contiguous 256-byte piece of its row
      uint4* out = reinterpret_cast<uint4*>(p.scores + (size_t)pair * kScoreTile + il * 128 + kh);
      const int32_t* se_tile = p.se + (size_t)row0 + kt * 128 + kh;
#pragma unroll
      for (int j = 0; j < 64; j += 4) {
        uint32_t v[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int jk = kt * 128 + kh + j + m;
          const bool vis = !part || (jk <= i && __ldg(se_tile + j + m) >= i);
          v[m] = vis ? order_key(acc[j + m]) : 0u;
        }
        out[j / 4] = make_uint4(v[0], v[1], v[2], v[3]);
      }
    }
  }

  __syncwarp();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == kIdxMma) tmem_dealloc(tmem, 512);
}


// One warp per query; a CTA holds eight consecutive queries of one query tile
// (longest lists first).  The query's candidates are its key rows in the
// tile pairs of its list (the scores' order keys, 0 where a key is not
// visible): one 512-byte row per key tile, a uint4 per lane, so every pass
// is one coalesced 16-byte load per lane and key tile, and after the first
// pass the rows come from L1/L2.  Byte-wise radix passes, most significant
// first, build the query's 256-bin histogram in shared memory and narrow the
// prefix of the k-th largest key; they stop as soon as every key left under
// the prefix is needed.  The emit pass walks the list in ascending key
// order: keys above the prefix, then the ones equal to it until the k are
// complete (ties to the smaller key index), their output offsets from warp
// prefix sums.
constexpr int kSelWarps = 8;
constexpr int kSelBatch = 8;    // key tiles whose rows one lane has in flight

template <typename F>
__device__ __forceinline__ void for_rows(const uint32_t* base, int cnt, int lane, F&& f) {
  for (int e0 = 0; e0 < cnt; e0 += kSelBatch) {
    uint4 v[kSelBatch];
#pragma unroll
    for (int u = 0; u < kSelBatch; ++u)
      if (e0 + u < cnt) v[u] = __ldg(reinterpret_cast<const uint4*>(base + (size_t)(e0 + u) * kScoreTile) + lane);
#pragma unroll
    for (int u = 0; u < kSelBatch; ++u)
      if (e0 + u < cnt) f(e0 + u, v[u]);
  }
}

__global__ void __launch_bounds__(kSelWarps * 32) index_select_kernel(const IdxParams p) {
  __shared__ __align__(16) uint32_t hist_all[kSelWarps * 256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kPerTile = 128 / kSelWarps;   // CTAs per query tile
  const int qt = p.NT - 1 - (int)(blockIdx.x / (p.R * kPerTile));
  const int r = (int)(blockIdx.x / kPerTile % p.R);
  const int il = (int)(blockIdx.x % kPerTile) * kSelWarps + warp, i = qt * 128 + il;
  uint32_t* hist = hist_all + warp * 256;
  const int cnt = p.csr_cnt[(size_t)r * p.NT + qt];
  const int32_t* list = p.csr + ((size_t)r * p.NT + qt) * p.NT;
  const int64_t pbase = (int64_t)p.row_base[r] + p.csr_off[(size_t)r * p.NT + qt];
  const int k = p.top_k;
  int32_t* oi = p.out_idx + ((size_t)r * p.T + i) * k;
  float* os = p.out_score + ((size_t)r * p.T + i) * k;
  if (cnt <= 0 || cnt > p.NT || pbase + cnt > p.cap) {   // uniform over the CTA
    if (threadIdx.x == 0) atomicOr(p.err, cnt <= 0 || cnt > p.NT ? kErrBadList : kErrCapacity);
    for (int n = lane; n < k; n += 32) {
      oi[n] = -1;
      os[n] = -INFINITY;
    }
    return;
  }
  const uint32_t* base = p.scores + (size_t)pbase * kScoreTile + (size_t)il * 128;

  // Candidates of a pass: visible keys (key != 0) whose masked bits equal the
  // prefix.  After the passes, "all" (at most k visible keys) is the prefix 0
  // under a full mask: then every visible key counts as above it.
  uint32_t prefix = 0, mask = 0;
  int rem = k;
#pragma unroll 1
  for (int d = 3; d >= 0; --d) {
    const int sh = 8 * d;
#pragma unroll
    for (int b = 0; b < 8; b += 4) *reinterpret_cast<uint4*>(hist + lane * 8 + b) = make_uint4(0u, 0u, 0u, 0u);
    __syncwarp();
    for_rows(base, cnt, lane, [&](int, const uint4& v) {
      const uint32_t key[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int m = 0; m < 4; ++m)
        if ((key[m] & mask) == prefix && key[m]) atomicAdd(&hist[(key[m] >> sh) & 255u], 1u);
    });
    __syncwarp();
    // lane holds bins 8 lane .. 8 lane + 7; count the keys in the bins of the lanes above
    uint32_t c8[8];
    int s = 0;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      c8[b] = hist[lane * 8 + b];
      s += (int)c8[b];
    }
    int incl = s;   // keys in the bins of this lane and the lanes above it
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_down_sync(0xffffffffu, incl, o);
      if (lane + o < 32) incl += t;
    }
    const int above = incl - s;
    if (d == 3 && __shfl_sync(0xffffffffu, incl, 0) <= k) {   // at most k visible keys: take them all
      prefix = 0;
      mask = 0xffffffffu;
      break;
    }
    // the lane whose range holds the rem-th largest key picks the bin
    const bool mine = above < rem && rem <= above + s;
    int bin = 0, cum = above, cb = 0;
    if (mine) {
#pragma unroll
      for (int b = 7; b >= 0; --b) {
        if (cum + (int)c8[b] >= rem) {
          bin = lane * 8 + b;
          cb = (int)c8[b];
          break;
        }
        cum += (int)c8[b];
      }
    }
    const int src = __ffs(__ballot_sync(0xffffffffu, mine)) - 1;
    bin = __shfl_sync(0xffffffffu, bin, src);
    cum = __shfl_sync(0xffffffffu, cum, src);
    cb = __shfl_sync(0xffffffffu, cb, src);
    prefix |= (uint32_t)bin << sh;
    mask |= 255u << sh;
    rem -= cum;
    if (cb == rem) break;   // every key under the prefix is taken
    __syncwarp();           // the bins were read before the next pass clears them
  }

  // emit in ascending key order; lane holds keys 4 lane .. 4 lane + 3 of each tile
  int n_out = 0, ties = 0;
  for_rows(base, cnt, lane, [&](int e, const uint4& v) {
    const uint32_t key[4] = {v.x, v.y, v.z, v.w};
    bool gt[4], eq[4];
    int ne = 0;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const uint32_t km = key[m] & mask;
      gt[m] = km > prefix;                   // above the prefix (0 never is)
      eq[m] = km == prefix && key[m] != 0u;  // under it: a tie candidate
      ne += eq[m];
    }
    // ties before this lane (inclusive scan of ne over lanes)
    int tin = ne;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, tin, o);
      if (lane >= o) tin += t;
    }
    int trank = ties + tin - ne;
    bool take[4];
    int nt = 0;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      take[m] = gt[m] || (eq[m] && trank < rem);
      trank += eq[m];
      nt += take[m];
    }
    ties += __shfl_sync(0xffffffffu, tin, 31);
    int pin = nt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, pin, o);
      if (lane >= o) pin += t;
    }
    int at = n_out + pin - nt;
    const int kt = list[e] >> 1;
#pragma unroll
    for (int m = 0; m < 4; ++m)
      if (take[m]) {
        oi[at] = kt * 128 + lane * 4 + m;
        os[at] = key_value(key[m]);
        ++at;
      }
    n_out += __shfl_sync(0xffffffffu, pin, 31);
  });
  for (int n = n_out + lane; n < k; n += 32) {
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
  *ws_bytes = 256 + (size_t)cap * kScoreTile * sizeof(uint32_t);
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
  p.scores = reinterpret_cast<uint32_t*>(static_cast<char*>(d_ws) + 256);
  p.out_idx = topk_idx;
  p.out_score = topk_score;
  const int64_t rows = (int64_t)desc->n_rows * desc->row_len;
  CUtensorMap mq, mk;
  if (!make_map_d(&mq, q, rows, p.H, p.D) || !make_map_d(&mk, k, rows, 1, p.D))
    return fail(STP_ECUDA, "stp_index_topk: tensor map encoding failed");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(p.err, 0, 4, s);
  const int smem = p.H * 128 * p.D * 2 + 2 * 128 * p.D * 2 + kIdxSmallBytes;
  static bool attr = false;
  if (e == cudaSuccess && !attr) {
    e = cudaFuncSetAttribute(index_scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kIdxQBytesMax + 2 * 128 * 128 * 2 + kIdxSmallBytes);
    attr = e == cudaSuccess;
  }
  if (e != cudaSuccess) return fail(STP_ECUDA, "stp_index_topk: %s", cudaGetErrorString(e));
  const unsigned grid = (unsigned)(NT * desc->n_rows);
  p.splits = (NT + kIdxPiece - 1) / kIdxPiece;
  index_scores_kernel<<<grid * p.splits, kIdxThreads, smem, s>>>(mq, mk, p);
  index_select_kernel<<<grid * (128 / kSelWarps), kSelWarps * 32, 0, s>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(STP_ECUDA, "stp_index_topk: %s", cudaGetErrorString(e));
  return STP_OK;
}
