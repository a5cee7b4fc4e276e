// Next-token log-probabilities over packed rows ("Prefix tree packing",
// tree-build section: the join copy keeps every trainable token's
// predecessor right before it in the same row; materialization section:
// loss_mask marks those predecessors).  For every position x with
// loss_mask[x] = 1:
//
//   logprob[x] = h[x] . W[tok[x + 1]] - ln sum_v exp(h[x] . W[v])
//
// and 0 elsewhere, without materializing the [positions, vocab] logits.
//
// logprob_tiles_kernel lists the 128-position tiles that hold a loss position
// and checks every loss position's target.  logprob_tc_kernel is persistent
// (one CTA per SM); its work units are (vocabulary split j, listed tile a),
// ordered so that the CTAs running at one time share the vocabulary rows they
// stream and hold few tiles of hidden states (unit_of).  Per unit, warp 4
// streams 64-wide hidden chunks of the tile (A) and of 256 vocabulary rows (B)
// through a four-stage TMA ring (rows past the vocabulary arrive as zeros);
// warp 5 issues tcgen05 MMAs (M = 128, N = 256) into one of two 256-column
// TMEM buffers per vocabulary tile; warps 0-3 (thread = position = TMEM lane)
// keep an online max / sum of exp over the logits and pick the target logit,
// while the tensor core fills the other buffer.  Each unit writes
// (max, sum, target logit) per position; logprob_combine_kernel merges the
// splits of a position into its log-probability.
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

constexpr int kLpThreads = 192;             // warps 0-3 epilogue, 4 TMA, 5 MMA
constexpr int kLpN = 256;                   // vocabulary rows per tile
constexpr int kLpStages = 4;
constexpr int kLpABytes = 128 * 64 * 2;     // 128 positions x 64 hidden
constexpr int kLpBBytes = kLpN * 64 * 2;    // 256 vocabulary rows x 64 hidden
constexpr int kLpStageBytes = kLpABytes + kLpBBytes;
constexpr int kLpSmem = kLpStages * kLpStageBytes + 1024 + 256;
constexpr int kLpMaxSplits = 64;
// Listed tiles per block of the unit order (see unit_of); 24 measured best of
// 12..76 on the 16384-position row (a 1.2 GB vocabulary projection).
constexpr int kLpTileBlock = 24;
constexpr float kLog2eLp = 1.4426950408889634f;
constexpr float kLn2Lp = 0.6931471805599453f;

struct LpParams {
  int N, T, Dh, V, n_vt, S, n_tiles, TA;
  const int32_t* tok;   // [N]
  const uint8_t* mask;  // [N]
  int32_t* n_act;       // number of listed tiles
  int32_t* act;         // [n_tiles] tile of each list slot
  int32_t* slot;        // [n_tiles] list slot of each tile, -1 when it holds no loss position
  float* part_m;        // [S][n_tiles][128] max logit of the unit (natural-log units)
  float* part_l;        // [S][n_tiles][128] sum of exp(logit - max)
  float* part_t;        // [S][n_tiles][128] target logit, -inf when outside the split
  float* out;           // [N]
  uint32_t* err;
};

enum { L_SF = 0, L_SE = 4, L_TF = 8, L_TE = 10, L_DRAIN = 12, L_COUNT = 13 };

typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                             const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                             CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_lp() {
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

// [rows, D] bf16 as a 2-D tensor (d, row); boxes of 64 d x box_rows rows,
// 128-byte swizzled; rows past the end read as zero.
bool make_map_rows(CUtensorMap* m, const void* base, int64_t rows, int D, int box_rows) {
  EncodeFn enc = encode_lp();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

// Unit u -> (vocabulary split j, list slot a).  The listed tiles are cut into
// blocks of TA; within a block the units run split-major.  The CTAs resident
// at one time then hold about TA tiles of hidden states (re-read from L2 for
// every vocabulary tile) and a few splits' vocabulary rows (shared by the TA
// CTAs of a split), which keeps both inside L2.
__device__ __forceinline__ void unit_of(const LpParams& p, int n_act, int u, int& j, int& a) {
  const int blk = p.TA * p.S;
  const int ab = u / blk, ul = u - ab * blk;
  const int rem = n_act - ab * p.TA;
  const int sz = rem < p.TA ? rem : p.TA;
  j = ul / sz;
  a = ab * p.TA + (ul - j * sz);
}

// One block of 128 threads per tile: lists the tile when it holds a loss
// position and checks each loss position's target (inside its row, in range).
__global__ void logprob_tiles_kernel(const LpParams p) {
  const int tile = blockIdx.x, x = tile * 128 + threadIdx.x;
  const bool on = p.mask[x] != 0;
  if (on) {
    const bool in_row = (x % p.T) != p.T - 1;
    const int t = in_row ? p.tok[x + 1] : -1;
    if (t < 0 || t >= p.V) atomicOr(p.err, kErrBadList);
  }
  if (__syncthreads_or(on)) {
    if (threadIdx.x == 0) {
      const int s = atomicAdd(p.n_act, 1);
      p.act[s] = tile;
      p.slot[tile] = s;
    }
  } else if (threadIdx.x == 0) {
    p.slot[tile] = -1;
  }
}

__global__ void __launch_bounds__(kLpThreads, 1)
    logprob_tc_kernel(const __grid_constant__ CUtensorMap th, const __grid_constant__ CUtensorMap tw,
                      const LpParams p) {
  extern __shared__ uint8_t smem_dyn[];
  // the 128-byte swizzle wants 1024-byte aligned stages
  uint8_t* smem_raw =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  const uint32_t big_s = smem_u32(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw + kLpStages * kLpStageBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + L_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_act = *p.n_act;
  const int units = n_act * p.S;
  if ((int)blockIdx.x >= units) return;   // uniform over the CTA
  const int n_kc = p.Dh / 64;

  if (threadIdx.x == 0) {
    for (int b = 0; b < L_COUNT; ++b) mbar_init(&bars[b], (b == L_TE || b == L_TE + 1) ? 4 : 1);
    *abort_flag = 0;
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

  if (warp == 4) {
    if (lane == 0) {
      // ------------------------------------------------------------ loads
      tma_prefetch_desc(&th);
      tma_prefetch_desc(&tw);
      int it = 0, last_phase[kLpStages] = {-1, -1, -1, -1};
      bool ok = true;
      for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
        int j, a;
        unit_of(p, n_act, u, j, a);
        const int x0 = p.act[a] * 128;
        const int vt1 = (j + 1) * p.n_vt / p.S;
        for (int vt = j * p.n_vt / p.S; ok && vt < vt1; ++vt)
          for (int kc = 0; kc < n_kc; ++kc, ++it) {
            const int st = it % kLpStages, n = it / kLpStages;
            if (it >= kLpStages && !mbar_wait(&bars[L_SE + st], (n - 1) & 1, abort_flag, p.err)) {
              ok = false;
              break;
            }
            uint8_t* dst = smem_raw + st * kLpStageBytes;
            mbar_expect_tx(&bars[L_SF + st], kLpStageBytes);
            tma_load_2d(dst, &th, &bars[L_SF + st], kc * 64, x0);
            tma_load_2d(dst + kLpABytes, &tw, &bars[L_SF + st], kc * 64, vt * kLpN);
            last_phase[st] = n & 1;
          }
      }
      for (int st = 0; st < kLpStages; ++st)
        if (last_phase[st] >= 0) mbar_wait_drain(&bars[L_SF + st], last_phase[st]);
    }
    __syncwarp();
  } else if (warp == 5) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA
      constexpr uint32_t idesc = idesc_bf16(128, kLpN, 0, 0);
      int it = 0, g = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
        int j, a;
        unit_of(p, n_act, u, j, a);
        const int vt1 = (j + 1) * p.n_vt / p.S;
        for (int vt = j * p.n_vt / p.S; ok && vt < vt1; ++vt, ++g) {
          const int b = g & 1;
          if (g >= 2 && !mbar_wait(&bars[L_TE + b], ((g >> 1) - 1) & 1, abort_flag, p.err)) {
            ok = false;
            break;
          }
          fence_after_sync();
          for (int kc = 0; kc < n_kc; ++kc, ++it) {
            const int st = it % kLpStages;
            if (!mbar_wait(&bars[L_SF + st], (it / kLpStages) & 1, abort_flag, p.err)) {
              ok = false;
              break;
            }
            fence_after_sync();
            const uint32_t a_lo = desc_lo_kmajor(big_s + st * kLpStageBytes);
            const uint32_t b_lo = desc_lo_kmajor(big_s + st * kLpStageBytes + kLpABytes);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ss_lo(tmem + b * kLpN, a_lo + kk * 2, b_lo + kk * 2, idesc, (kc > 0 || kk > 0) ? 1u : 0u);
            mma_commit(&bars[L_SE + st]);
          }
          if (ok) mma_commit(&bars[L_TF + b]);
        }
      }
      mma_commit(&bars[L_DRAIN]);
      mbar_wait_drain(&bars[L_DRAIN], 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    int g = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
      int j, a;
      unit_of(p, n_act, u, j, a);
      const int xr = p.act[a] * 128 + threadIdx.x;   // position = TMEM lane
      int target = -1;
      if (p.mask[xr] && (xr % p.T) != p.T - 1) {
        const int t = p.tok[xr + 1];
        if (t >= 0 && t < p.V) target = t;
      }
      float m = -INFINITY, l = 0.f, tl = -INFINITY;   // in log2 units: logit * log2(e)
      const int vt1 = (j + 1) * p.n_vt / p.S;
      for (int vt = j * p.n_vt / p.S; vt < vt1; ++vt, ++g) {
        const int b = g & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&bars[L_TF + b], (g >> 1) & 1, abort_flag, p.err))) {
          ok = false;
          break;
        }
        fence_after_sync();
#pragma unroll 1
        for (int c = 0; c < kLpN / 64; ++c) {
          uint32_t x[64];
          tmem_ld32(tmem + lane_base + b * kLpN + c * 64, x);
          tmem_ld32(tmem + lane_base + b * kLpN + c * 64 + 32, x + 32);
          tmem_ld_wait();
          const int vc = vt * kLpN + c * 64;
          const int lim = p.V - vc;   // columns at or past it lie outside the vocabulary
          float cm = -INFINITY;
#pragma unroll
          for (int q = 0; q < 64; ++q) {
            const float y = q < lim ? __uint_as_float(x[q]) * kLog2eLp : -INFINITY;
            x[q] = __float_as_uint(y);
            cm = fmaxf(cm, y);
          }
          const int d = target - vc;
          if ((unsigned)d < 64u) {
#pragma unroll
            for (int q = 0; q < 64; ++q)
              if (q == d) tl = __uint_as_float(x[q]);
          }
          const float mn = fmaxf(m, cm);   // finite: column 0 of a tile lies inside the vocabulary
          float s0 = 0.f, s1 = 0.f;
#pragma unroll
          for (int q = 0; q < 64; q += 2) {
            s0 += ex2(__uint_as_float(x[q]) - mn);
            s1 += ex2(__uint_as_float(x[q + 1]) - mn);
          }
          l = l * ex2(m - mn) + (s0 + s1);
          m = mn;
        }
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[L_TE + b]);
      }
      if (!ok) break;
      const size_t at = ((size_t)j * p.n_tiles + a) * 128 + threadIdx.x;
      p.part_m[at] = m * kLn2Lp;
      p.part_l[at] = l;
      p.part_t[at] = tl * kLn2Lp;
    }
  }

  __syncwarp();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == 5) tmem_dealloc(tmem, 512);
}

// One thread per position: merges the S partials of a loss position.
__global__ void logprob_combine_kernel(const LpParams p) {
  const int x = blockIdx.x * blockDim.x + threadIdx.x;
  if (x >= p.N) return;
  const int a = p.slot[x >> 7];
  if (!p.mask[x] || a < 0) {
    p.out[x] = 0.f;
    return;
  }
  const size_t base = (size_t)a * 128 + (x & 127), stride = (size_t)p.n_tiles * 128;
  float M = -INFINITY, t = -INFINITY;
  for (int j = 0; j < p.S; ++j) {
    M = fmaxf(M, p.part_m[base + j * stride]);
    t = fmaxf(t, p.part_t[base + j * stride]);
  }
  float L = 0.f;
  for (int j = 0; j < p.S; ++j) L += p.part_l[base + j * stride] * expf(p.part_m[base + j * stride] - M);
  p.out[x] = t - (M + logf(L));
}

int lp_splits(int n_vt) { return n_vt < kLpMaxSplits ? n_vt : kLpMaxSplits; }

struct LpLayout {
  size_t n_act, act, slot, part, total;
};

// The error word sits at offset 0 and the tile count at 256; both are
// cleared before each call.
LpLayout lp_layout(int64_t N, int S) {
  const int64_t n_tiles = N / 128;
  LpLayout L;
  size_t o = 512;
  L.n_act = 256;
  L.act = o;
  o += align256((size_t)n_tiles * 4);
  L.slot = o;
  o += align256((size_t)n_tiles * 4);
  L.part = o;
  o += 3 * align256((size_t)S * N * 4);
  L.total = o;
  return L;
}

stp_status check_lp(const stp_logprob_desc* d) {
  if (!d) return fail(STP_EINVAL, "logprob descriptor is NULL");
  if (d->n_rows < 0 || d->row_len <= 0 || d->row_len % kTile)
    return fail(STP_EINVAL, "need n_rows >= 0 and row_len a positive multiple of 128");
  if (d->hidden < 64 || d->hidden % 64 || d->hidden > 16384)
    return fail(STP_EUNSUPPORTED, "hidden must be a multiple of 64 in [64, 16384] (got %d)", d->hidden);
  if (d->vocab < 1 || d->vocab > (1 << 24)) return fail(STP_EUNSUPPORTED, "vocab must lie in [1, 2^24]");
  if ((int64_t)d->n_rows * d->row_len > (1 << 28)) return fail(STP_EUNSUPPORTED, "more than 2^28 positions");
  return STP_OK;
}

}  // namespace
}  // namespace stp

using namespace stp;

extern "C" stp_status stp_logprob_workspace_size(const stp_logprob_desc* desc, size_t* ws_bytes) {
  clear_error();
  stp_status st = check_lp(desc);
  if (st) return st;
  if (!ws_bytes) return fail(STP_EINVAL, "stp_logprob_workspace_size: NULL output");
  const int n_vt = (desc->vocab + kLpN - 1) / kLpN;
  *ws_bytes = lp_layout((int64_t)desc->n_rows * desc->row_len, lp_splits(n_vt)).total;
  return STP_OK;
}

extern "C" stp_status stp_logprob_gather(const stp_logprob_desc* desc, const void* hidden, const void* w_vocab,
                                         const int32_t* d_token_ids, const uint8_t* d_loss_mask,
                                         float* logprob, void* d_ws, void* stream) {
  clear_error();
  stp_status st = check_lp(desc);
  if (st) return st;
  if (!hidden || !w_vocab || !d_token_ids || !d_loss_mask || !logprob || !d_ws)
    return fail(STP_EINVAL, "stp_logprob_gather: NULL device pointer");
  if ((reinterpret_cast<uintptr_t>(hidden) | reinterpret_cast<uintptr_t>(w_vocab)) & 15 ||
      reinterpret_cast<uintptr_t>(d_ws) & 255)
    return fail(STP_EINVAL, "stp_logprob_gather: hidden and w_vocab 16-byte, ws 256-byte aligned");
  if (desc->n_rows == 0) return STP_OK;
  const int N = desc->n_rows * desc->row_len;
  LpParams p;
  p.N = N;
  p.T = desc->row_len;
  p.Dh = desc->hidden;
  p.V = desc->vocab;
  p.n_vt = (desc->vocab + kLpN - 1) / kLpN;
  p.S = lp_splits(p.n_vt);
  p.n_tiles = N / 128;
  p.TA = kLpTileBlock;
  p.tok = d_token_ids;
  p.mask = d_loss_mask;
  char* ws = static_cast<char*>(d_ws);
  const LpLayout L = lp_layout(N, p.S);
  const size_t part = align256((size_t)p.S * N * 4);
  p.err = reinterpret_cast<uint32_t*>(ws);
  p.n_act = reinterpret_cast<int32_t*>(ws + L.n_act);
  p.act = reinterpret_cast<int32_t*>(ws + L.act);
  p.slot = reinterpret_cast<int32_t*>(ws + L.slot);
  p.part_m = reinterpret_cast<float*>(ws + L.part);
  p.part_l = reinterpret_cast<float*>(ws + L.part + part);
  p.part_t = reinterpret_cast<float*>(ws + L.part + 2 * part);
  p.out = logprob;
  CUtensorMap mh, mw;
  if (!make_map_rows(&mh, hidden, N, p.Dh, 128) || !make_map_rows(&mw, w_vocab, p.V, p.Dh, kLpN))
    return fail(STP_ECUDA, "stp_logprob_gather: tensor map encoding failed");
  int dev = 0, n_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(logprob_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kLpSmem);
  });
  if (e == cudaSuccess) e = attr_err;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws, 0, 512, s);
  if (e != cudaSuccess) return fail(STP_ECUDA, "stp_logprob_gather: %s", cudaGetErrorString(e));
  const int units_max = p.n_tiles * p.S;
  const int grid = units_max < n_sm ? units_max : n_sm;
  logprob_tiles_kernel<<<(unsigned)p.n_tiles, 128, 0, s>>>(p);
  logprob_tc_kernel<<<(unsigned)grid, kLpThreads, kLpSmem, s>>>(mh, mw, p);
  logprob_combine_kernel<<<(unsigned)((N + 255) / 256), 256, 0, s>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(STP_ECUDA, "stp_logprob_gather: %s", cudaGetErrorString(e));
  return STP_OK;
}
