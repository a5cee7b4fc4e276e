// Tree attention on the tcgen05 tensor cores (bf16 in, f32 accumulate,
// head_dim 128), driven by the tile lists of stp_classify.
//
// Forward ("Prefix tree packing", attention section; masked causal attention
// with FlashAttention-style online softmax).  One CTA per (row, kv head,
// query tile, pair of query heads of the kv head's group): both heads read
// the same key/value tiles, so one TMA load of K and V feeds two query tiles.
//   warp 8      TMA producer: Q tiles once, then K / V tiles of the query
//               tile's list through a 2-stage ring;
//   warp 9      MMA issuer: S_h = Q_h K^T (M=N=128, K=128) into TMEM, then
//               O_h += P_h V (P_h read from TMEM, V an MN-major operand);
//               owns the TMEM allocation (512 columns: S_0, S_1, O_0, O_1);
//   warps 0-3   softmax for head slot 0, warps 4-7 for head slot 1: one thread
//               per query row (= TMEM lane); the predicate
//               j <= i && subtree_end[j] >= i is applied on PARTIAL tiles only;
//               online softmax in base 2; O is rescaled in TMEM only when the
//               running max grows by more than 2^8 (exact: numerator and
//               denominator keep the same reference max).
// Each softmax group writes its P as packed bf16 pairs over the first 64
// columns of its own S; the MMA warp issues PV_0(e), S_0(e+1), PV_1(e),
// S_1(e+1), so the tensor core works on one head while the other's softmax
// runs.
// Every mbarrier wait is bounded; a wait that runs out sets the workspace
// error word, the CTA drains its outstanding copies and MMAs, frees TMEM and
// returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"
#include "layout.h"
#include "tc.h"
#include "tc_ptx.cuh"

namespace stp {
namespace {

using namespace tc;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

constexpr int kTileBytes = 128 * 128 * 2;  // one 128 x 128 bf16 tile
constexpr int kHalfTile = kTileBytes / 2;  // one 128-row x 64-column swizzled block
constexpr int kSmallBytes = 256;           // barriers, TMEM slot, abort flag
constexpr int kFwdBigBytes = 6 * kTileBytes;  // Q0 Q1 K0 K1 V0 V1
constexpr int kSmemLimit = 232448;

// ------------------------------------------------------------------------
// Host: tensor maps
// ------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// [rows, H, 128] bf16 viewed as a 3-D tensor (d, head, row); boxes of
// 64 d x 1 head x 128 rows land as 128 rows of 128 bytes, 128-byte swizzled.
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int H) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {128, (cuuint64_t)H, (cuuint64_t)rows};
  cuuint64_t strides[2] = {128 * 2, (cuuint64_t)H * 128 * 2};
  cuuint32_t box[3] = {64, 1, 128};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------------------
// Device helpers
// ------------------------------------------------------------------------

struct FwdParams {
  int R, T, Hq, Hkv, NT, G, npairs;
  float scale_log2;
  const int32_t* se;
  const int32_t* csr_cnt;
  const int32_t* csr;
  __nv_bfloat16* o;
  float* lse;
  uint32_t* err;
};

enum {
  B_Q = 0, B_KF = 1, B_VF = 3, B_KE = 5, B_VE = 7, B_SF = 9, B_PF = 11, B_OD = 13, B_DRAIN = 15,
  B_COUNT = 16
};

// Forward: 12 warps = three full warpgroups; registers move from the control
// warpgroup (TMA + MMA issue) to the two softmax warpgroups with setmaxnreg,
// at the head of each role's branch: 384 x 168 at launch = 256 x 216 + 128 x 72,
// and per SM sub-partition (warps w, w+4, w+8) 216 + 216 + 72 <= 512.
constexpr int kThreads = 384;
constexpr int kRegsAtLaunch = 168, kRegsMath = 216, kRegsCtl = 72;
static_assert(kThreads * kRegsAtLaunch >= 256 * kRegsMath + 128 * kRegsCtl, "register split");

__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + B_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t raw = smem_u32(smem_raw) + kSmallBytes;
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t* big = smem_raw + kSmallBytes + pad;
  const uint32_t big_s = raw + pad;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per_qt = p.R * p.Hkv * p.npairs;
  const int qt = p.NT - 1 - (int)(blockIdx.x / per_qt);
  int rem = blockIdx.x % per_qt;
  const int r = rem / (p.Hkv * p.npairs);
  rem %= p.Hkv * p.npairs;
  const int g = rem / p.npairs, pair = rem % p.npairs;
  const int h0 = g * p.G + 2 * pair;
  const int nh = min(2, p.G - 2 * pair);
  const int cnt = p.csr_cnt[(size_t)r * p.NT + qt];
  const int32_t* list = p.csr + ((size_t)r * p.NT + qt) * p.NT;
  const int row0 = r * p.T;  // first row of this packed row in the [R*T] views

  if (threadIdx.x == 0) {
    mbar_init(&bars[B_Q], 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars[B_KF + s], 1);
      mbar_init(&bars[B_VF + s], 1);
      mbar_init(&bars[B_KE + s], 1);
      mbar_init(&bars[B_VE + s], 1);
      mbar_init(&bars[B_SF + s], 1);
      mbar_init(&bars[B_PF + s], 4);  // one arrival per softmax warp
      mbar_init(&bars[B_OD + s], 1);
    }
    mbar_init(&bars[B_DRAIN], 1);
    *abort_flag = 0;
    if (pad + kSmallBytes + kFwdBigBytes > kSmemLimit || cnt <= 0 || cnt > p.NT) {
      *abort_flag = 1;
      atomicOr(p.err, cnt <= 0 || cnt > p.NT ? kErrBadList : kErrTmem);
    }
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const bool run = !*abort_flag;

  uint32_t q_s[2] = {big_s, big_s + kTileBytes};
  uint32_t k_s[2] = {big_s + 2 * kTileBytes, big_s + 3 * kTileBytes};
  uint32_t v_s[2] = {big_s + 4 * kTileBytes, big_s + 5 * kTileBytes};

  int issued_k[2] = {-1, -1};  // producer: last issued use of each stage
  int issued_v[2] = {-1, -1};

  if (warp >= 8) {
    regs_dec<kRegsCtl>();
  }
  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && run) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      mbar_expect_tx(&bars[B_Q], nh * kTileBytes);
      for (int hs = 0; hs < nh; ++hs)
        for (int hf = 0; hf < 2; ++hf)
          tma_load_3d(big + hs * kTileBytes + hf * kHalfTile, &tq, &bars[B_Q], hf * 64, h0 + hs,
                      row0 + qt * 128);
      for (int e = 0; e < cnt; ++e) {
        const int st = e & 1, n = e >> 1;
        const int kt = list[e] >> 1;
        if (kt < 0 || kt > qt) {
          *abort_flag = 1;
          atomicOr(p.err, kErrBadList);
          break;
        }
        // K and V of a later entry into L2 (see the backward producer)
        if (e + 2 < cnt) {
          const int kt2 = min(max(list[e + 2] >> 1, 0), p.NT - 1);
          for (int hf = 0; hf < 2; ++hf) {
            tma_prefetch_l2_3d(&tk, hf * 64, g, row0 + kt2 * 128);
            tma_prefetch_l2_3d(&tv, hf * 64, g, row0 + kt2 * 128);
          }
        }
        if (e >= 2 && !mbar_wait(&bars[B_KE + st], (n - 1) & 1, abort_flag, p.err)) break;
        mbar_expect_tx(&bars[B_KF + st], kTileBytes);
        for (int hf = 0; hf < 2; ++hf)
          tma_load_3d(big + (2 + st) * kTileBytes + hf * kHalfTile, &tk, &bars[B_KF + st],
                      hf * 64, g, row0 + kt * 128);
        issued_k[st] = n;
        if (e >= 2 && !mbar_wait(&bars[B_VE + st], (n - 1) & 1, abort_flag, p.err)) break;
        mbar_expect_tx(&bars[B_VF + st], kTileBytes);
        for (int hf = 0; hf < 2; ++hf)
          tma_load_3d(big + (4 + st) * kTileBytes + hf * kHalfTile, &tv, &bars[B_VF + st],
                      hf * 64, g, row0 + kt * 128);
        issued_v[st] = n;
      }
      // wait (bounded) for every copy this warp started
      mbar_wait_drain(&bars[B_Q], 0);
      for (int st = 0; st < 2; ++st) {
        if (issued_k[st] >= 0) mbar_wait_drain(&bars[B_KF + st], issued_k[st] & 1);
        if (issued_v[st] >= 0) mbar_wait_drain(&bars[B_VF + st], issued_v[st] & 1);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && run) {
      constexpr uint32_t idesc_s = idesc_bf16(128, 128, 0, 0);
      constexpr uint32_t idesc_o = idesc_bf16(128, 128, 0, 1);
      // descriptor low words; slice kk adds a constant to the start-address field
      const uint32_t q_km0 = desc_lo_kmajor(q_s[0]), q_km1 = desc_lo_kmajor(q_s[1]);
      const uint32_t k_km0 = desc_lo_kmajor(k_s[0]), v_mn0 = desc_lo_mnmajor(v_s[0]);
      constexpr uint32_t kStage = kTileBytes >> 4;
      auto km = [](int kk) { return (uint32_t)((kk >> 2) * (kHalfTile >> 4) + (kk & 3) * 2); };
      auto mn = [](int kk) { return (uint32_t)(kk * 128); };
      bool ok = mbar_wait(&bars[B_Q], 0, abort_flag, p.err) &&
                mbar_wait(&bars[B_KF], 0, abort_flag, p.err);
      if (ok) {
        fence_after_sync();
#pragma unroll
        for (int hs = 0; hs < 2; ++hs) {
          if (hs < nh) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ss_lo(tmem + hs * 128, (hs ? q_km1 : q_km0) + km(kk), k_km0 + km(kk), idesc_s, kk > 0);
            mma_commit(&bars[B_SF + hs]);
          }
        }
        mma_commit(&bars[B_KE]);
      }
#pragma unroll 1
      for (int e = 0; ok && e < cnt; ++e) {
        const int st = e & 1, n = e >> 1;
        const int st1 = (e + 1) & 1, n1 = (e + 1) >> 1;
        const uint32_t v_mn = v_mn0 + (st ? kStage : 0);
        const uint32_t k_next = k_km0 + (st1 ? kStage : 0);
        if (!mbar_wait(&bars[B_VF + st], n & 1, abort_flag, p.err)) break;
#pragma unroll
        for (int hs = 0; hs < 2; ++hs) {
          if (hs >= nh || !ok) continue;
          if (!mbar_wait(&bars[B_PF + hs], e & 1, abort_flag, p.err)) {
            ok = false;
            continue;
          }
          fence_after_sync();
          // O_hs += P_hs V: P_hs is packed bf16 in TMEM over the first 64
          // columns of S_hs
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts_lo(tmem + 256 + hs * 128, tmem + hs * 128 + kk * 8, v_mn + mn(kk), idesc_o, (e > 0 || kk > 0));
          mma_commit(&bars[B_OD + hs]);
          if (e + 1 < cnt) {
            if (hs == 0 && !mbar_wait(&bars[B_KF + st1], n1 & 1, abort_flag, p.err)) {
              ok = false;
              continue;
            }
            fence_after_sync();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ss_lo(tmem + hs * 128, (hs ? q_km1 : q_km0) + km(kk), k_next + km(kk), idesc_s, kk > 0);
            mma_commit(&bars[B_SF + hs]);
            if (hs == nh - 1) mma_commit(&bars[B_KE + st1]);
          }
        }
        if (ok) mma_commit(&bars[B_VE + st]);
      }
    }
    if (lane == 0 && run) {
      // wait (bounded) for every MMA this thread issued
      mma_commit(&bars[B_DRAIN]);
      mbar_wait_drain(&bars[B_DRAIN], 0);
    }
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax
    regs_inc<kRegsMath>();
    const int hs = warp >> 2;
    const int row = threadIdx.x & 127;
    const int i = qt * 128 + row;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t s_addr = tmem + lane_base + hs * 128;
    const uint32_t o_addr = tmem + lane_base + 256 + hs * 128;
    const int32_t* se_row = p.se + (size_t)row0;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = run && hs < nh;
    for (int e = 0; ok && e < cnt; ++e) {
      const int ent = list[e], kt = ent >> 1, part = ent & 1, k0 = kt * 128;
      // visibility bits of a partial tile (j <= i && subtree_end[j] >= i),
      // computed before the scores are ready so the loads stay off the
      // critical path
      uint32_t vis[4] = {~0u, ~0u, ~0u, ~0u};
      if (part) {
        const int4* se4 = reinterpret_cast<const int4*>(se_row + k0);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          uint32_t bits = 0;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const int4 v = __ldg(se4 + 8 * w + c);
            const int j = k0 + 32 * w + 4 * c;
            bits |= (uint32_t)(j + 0 <= i && v.x >= i) << (4 * c + 0);
            bits |= (uint32_t)(j + 1 <= i && v.y >= i) << (4 * c + 1);
            bits |= (uint32_t)(j + 2 <= i && v.z >= i) << (4 * c + 2);
            bits |= (uint32_t)(j + 3 <= i && v.w >= i) << (4 * c + 3);
          }
          vis[w] = bits;
        }
      }
      if (!__all_sync(0xffffffffu, mbar_wait(&bars[B_SF + hs], e & 1, abort_flag, p.err))) {
        ok = false;
        break;
      }
      fence_after_sync();
      // the whole score row: 128 TMEM columns of this thread's lane
      uint32_t u[128];
      tmem_ld32(s_addr + 0, u);
      tmem_ld32(s_addr + 32, u + 32);
      tmem_ld32(s_addr + 64, u + 64);
      tmem_ld32(s_addr + 96, u + 96);
      tmem_ld_wait();
      if (part) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (!((vis[c >> 5] >> (c & 31)) & 1u)) u[c] = 0xff800000u;
      }
      // row max on the raw scores (the scale is positive); four independent
      // chains keep the dependent-latency path short
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < 128; c += 8)
#pragma unroll
        for (int t = 0; t < 4; ++t)
          mx4[t] = max3(mx4[t], __uint_as_float(u[c + 2 * t]), __uint_as_float(u[c + 2 * t + 1]));
      const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      const float m_new = fmaxf(m_run, mx * p.scale_log2);
      const float m_use = (m_new > m_run + kRescaleThreshold) ? m_new : m_run;
      const float m_sub = (m_use == -INFINITY) ? 0.f : m_use;
      const float alpha = ex2(m_run - m_sub);
      // p = 2^(s * scale log2e - m), two columns per packed FFMA
      const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
      const float2 nm2 = make_float2(-m_sub, -m_sub);
      float2 acc2 = make_float2(0.f, 0.f);
      // P goes back over the first 64 score columns (already read), half a
      // row at a time.  PV of the previous tile, which read the old P and
      // wrote O, completed before this tile's S (issued after it), so both
      // may be overwritten now.
      float2 acc2b = make_float2(0.f, 0.f);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const int c0 = 64 * hf + 2 * c;
          const float2 y0 = __ffma2_rn(make_float2(__uint_as_float(u[c0]), __uint_as_float(u[c0 + 1])), sl2, nm2);
          const float2 y1 = __ffma2_rn(make_float2(__uint_as_float(u[c0 + 2]), __uint_as_float(u[c0 + 3])), sl2, nm2);
          const float2 p0 = make_float2(ex2(y0.x), ex2(y0.y));
          const float2 p1 = make_float2(ex2(y1.x), ex2(y1.y));
          acc2 = __fadd2_rn(acc2, p0);
          acc2b = __fadd2_rn(acc2b, p1);
          pk[c] = pack_bf16x2(p0.x, p0.y);
          pk[c + 1] = pack_bf16x2(p1.x, p1.y);
        }
        tmem_st32(s_addr + 32 * hf, pk);
      }
      const float rs = (acc2.x + acc2b.x) + (acc2.y + acc2b.y);
      if (e > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        uint32_t u[32];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          tmem_ld32(o_addr + c * 32, u);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 32; ++k) u[k] = __float_as_uint(__uint_as_float(u[k]) * alpha);
          tmem_st32(o_addr + c * 32, u);
        }
      }
      tmem_st_wait();
      l_run = l_run * alpha + rs;
      m_run = m_use;
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_PF + hs]);
    }
    if (ok && mbar_wait(&bars[B_OD + hs], (cnt - 1) & 1, abort_flag, p.err)) {
      fence_after_sync();
      const int h = h0 + hs;
      __nv_bfloat16* orow = p.o + (((size_t)row0 + i) * p.Hq + h) * 128;
      const float inv = 1.f / l_run;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t u[32];
        tmem_ld32(o_addr + c * 32, u);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint4 v;
          v.x = pack_bf16x2(__uint_as_float(u[8 * k + 0]) * inv, __uint_as_float(u[8 * k + 1]) * inv);
          v.y = pack_bf16x2(__uint_as_float(u[8 * k + 2]) * inv, __uint_as_float(u[8 * k + 3]) * inv);
          v.z = pack_bf16x2(__uint_as_float(u[8 * k + 4]) * inv, __uint_as_float(u[8 * k + 5]) * inv);
          v.w = pack_bf16x2(__uint_as_float(u[8 * k + 6]) * inv, __uint_as_float(u[8 * k + 7]) * inv);
          *reinterpret_cast<uint4*>(orow + c * 32 + 8 * k) = v;
        }
      }
      p.lse[((size_t)r * p.Hq + h) * p.T + i] = (m_run + log2f(l_run)) * kLn2;
    }
  }

  // ---------------------------------------------------------------- teardown
  __syncwarp();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == 9) tmem_dealloc(tmem, 512);
}


// ------------------------------------------------------------------------
// Backward
// ------------------------------------------------------------------------
//
// Two kernels after the Delta pass.
//
// bwd_tc_kernel, one CTA per (row r, kv head g, key tile kt): the key tile's
// list of non-empty query tiles, times the G query heads of the group, gives
// the iterations j = (query tile, head).  dK and dV accumulate in TMEM over
// all iterations; each iteration's dS^T tile also goes out to the workspace
// slot of its (pair, head), for the dQ kernel.
// Tensor memory (512 columns, keys on lanes):
//   0..127    S^T = K Q^T (f32);
//   128..255  dP^T = V dO^T (f32); once read, P^T and dS^T as packed bf16
//             pairs: per 64-query half, P^T over its first 32 columns and
//             dS^T over the next 32;
//   256..383  dV += P^T dO (A from TMEM);  384..511  dK += dS^T Q (A from TMEM).
// The row terms of the softmax backward ride on the tensor core: one more
// K = 16 slice per product, a column of ones against a bias tile, adds
// -LSE_i / scale to every score of query i and -Delta_i to every dP, so the
// elementwise pass needs no per-query constants (p = 2^(s' scale log2e),
// dS = p dP'); each bias is split into three bf16 terms (hi + mid + lo,
// about 24 significant bits), written per query tile by the Delta pass.
// The S^T columns are free as soon as the elementwise pass has loaded them,
// so S^T of the iteration after next is computed while that pass runs, and
// the tensor core's order is dK(j), dV(j), dP^T(j+1), S^T(j+2): the pass of
// j+1 starts with its scores already in TMEM, computes its exponentials
// while dK(j) and dV(j) run, and waits only for dP^T(j+1).  Neither P^T nor
// dS^T goes through shared memory (next to MMAs whose operands are both in
// shared memory, shared-memory stores wait hundreds of cycles each), and the
// elementwise warps do not store dS^T to global memory either: a store
// warpgroup copies it from TMEM to the workspace while the next pass runs.
// 16 warps:
//   warps 0-7   elementwise, one thread per key (= TMEM lane); warps 0-3 take
//               query columns 0..63, warps 4-7 columns 64..127:
//               p = 2^(s' scale log2e) (masked on PARTIAL tiles with the
//               thread's own subtree_end[j]), then once dP^T(j) is in TMEM
//               dS = p dP'; P^T and dS^T back to TMEM;
//   warp 8      TMA: K, V once; Q with its score bias tile and dO with its dP
//               bias tile, per iteration, through two 2-stage rings;
//   warp 9      MMA issue and TMEM owner;
//   warps 10-11 no role (a full warpgroup for the register split);
//   warps 12-15 dS^T store: TMEM -> registers -> the (pair, head) slot, in a
//               layout where each warp's 16-byte stores are contiguous.
// dK (times scale) and dV leave TMEM once at the end.
//
// dS^T tile layout in the workspace (bf16, 32 KiB per (pair, head)): 16
// blocks of 2048 bytes, block c holding query columns 8c..8c+7 of all 128
// keys, 16 bytes per key: byte offset c * 2048 + key * 16.  As an MMA
// operand with the queries as M (the dQ product) that is the no-swizzle
// MN-major layout: 8 x 16-byte core matrices, 2048 bytes apart along the
// queries and 128 bytes apart along the keys.
//
// dq_tc_kernel, one CTA per (row, kv head, query tile, up to four query heads
// of the group): dQ_h = scale sum over the query tile's key tiles of dS K, the
// dS tiles read back from the workspace and K by TMA, accumulated in TMEM
// (128 columns per head).  Every dQ element is summed in one fixed order, and
// no atomics are involved.
//
// The kv heads run in groups, each on its own stream (bwd_tc_kernel then
// dq_tc_kernel); a group's dS tiles live in one of `slots` workspace slots,
// and a group that reuses a slot waits for the dQ pass of the group before it.

struct BwdParams {
  int R, T, Hq, Hkv, NT, G;
  int g0, ng;           // kv heads [g0, g0 + ng) of this launch
  int slot_heads;       // query heads per pair in a dS slot
  float scale_log2;
  int64_t cap;          // dS pairs per slot
  const int32_t* se;
  const int32_t* csc_cnt;
  const int32_t* csc;
  const int32_t* csc_pair;
  const uint8_t* sbias; // [R][Hq][NT] bias tiles of the scores (-LSE / scale)
  const uint8_t* dbias; // [R][Hq][NT] bias tiles of dP (-Delta)
  uint8_t* ds;          // this launch's slot: [pair][slot_heads] dS^T tiles
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  float scale;
  uint32_t* err;
};

enum {
  C_KV = 0, C_QF = 1, C_QE = 3, C_DF = 5, C_DE = 7, C_SF = 9, C_SR = 10, C_DPF = 11, C_DR = 12, C_DSR = 13,
  C_DONE = 14, C_DRAIN = 15, C_COUNT = 16
};
// shared memory: [K | V | Q0 | Q1 | dO0 | dO1] (1024-aligned, at the start of
// dynamic shared memory) [SB0 | SB1 | DB0 | DB1 | ONES] (4 KiB each: bias
// tiles of the two ring stages, and the ones operand) [barriers ...]
constexpr int kBwdBigBytes = 6 * kTileBytes;
constexpr int kBwdBiasBytes = 5 * (int)kBiasTileBytes;
constexpr int kBwdSmem = kBwdBigBytes + kBwdBiasBytes + kSmallBytes;
static_assert(kBwdSmem <= kSmemLimit, "backward shared memory");
constexpr int kDsBlock = 128 * 16;  // one 8-query block of a dS^T tile: 16 bytes per key

// Bias tile and ones operand: [128 rows][16] bf16, K-major without swizzle:
// 8 x 16-byte core matrices, 128 bytes apart along K (leading-dimension
// offset) and 256 bytes apart along the rows (stride-dimension offset); row
// q, column k at byte (q / 8) 256 + (k / 8) 128 + (q % 8) 16 + (k % 8) 2.
__device__ __forceinline__ uint64_t bias_desc(uint32_t addr) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(128u >> 4) << 16) | ((uint64_t)(256u >> 4) << 32) |
         (1ull << 46);
}
// 16 warps x 128 registers at launch, rebalanced with setmaxnreg:
// 128 x (192 + 192 (elementwise) + 56 (control) + 72 (store)) = 65536, and per
// SM sub-partition (warps w, w+4, w+8, w+12) 512.
constexpr int kBwdThreads = 512;
constexpr int kBwdPrefetch = 2;  // iterations ahead for the L2 prefetch of Q, dO
constexpr int kBwdRegsMath = 192, kBwdRegsCtl = 56, kBwdRegsStore = 72;
static_assert(128 * (2 * kBwdRegsMath + kBwdRegsCtl + kBwdRegsStore) <= kBwdThreads * 128, "register split");

__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                  const BwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* big = smem_raw;
  const uint32_t big_s = smem_u32(smem_raw);
  uint8_t* bias = smem_raw + kBwdBigBytes;   // SB0 SB1 DB0 DB1 ONES
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw + kBwdBigBytes + kBwdBiasBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t k_s = big_s, v_s = big_s + kTileBytes;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per_kt = p.R * p.ng;
  const int kt = (int)(blockIdx.x / per_kt);
  const int r = (blockIdx.x % per_kt) / p.ng;
  const int gl = (int)(blockIdx.x % p.ng);  // kv head within this launch
  const int g = p.g0 + gl;
  const int cnt = p.csc_cnt[(size_t)r * p.NT + kt];
  const int32_t* list = p.csc + ((size_t)r * p.NT + kt) * p.NT;
  const int32_t* pairs = p.csc_pair + ((size_t)r * p.NT + kt) * p.NT;
  const int n_it = cnt * p.G;
  const int row0 = r * p.T;

  if (threadIdx.x == 0) {
    for (int b = 0; b < C_COUNT; ++b)
      // C_SR, C_DR: one arrival per elementwise warp; C_DSR: per store warp
      mbar_init(&bars[b], (b == C_SR || b == C_DR) ? 8 : (b == C_DSR ? 4 : 1));
    *abort_flag = 0;
    if ((big_s & 1023u) != 0 || cnt <= 0 || cnt > p.NT) {
      *abort_flag = 1;
      atomicOr(p.err, (big_s & 1023u) != 0 ? kErrTmem : kErrBadList);
    }
    fence_mbar_init();
  }
  {
    // the ones operand [128 keys][16]: 1 in columns 0-2 (bias tile layout)
    const int e = threadIdx.x;  // one 16-byte row chunk per thread: 256 chunks
    if (e < 256) {
      const int key = e >> 1, kc = e & 1;
      const uint32_t one = 0x3F80u;  // bf16 1.0
      const uint4 v = kc ? make_uint4(0u, 0u, 0u, 0u) : make_uint4(one | (one << 16), one, 0u, 0u);
      *reinterpret_cast<uint4*>(bias + 4 * kBiasTileBytes + (key >> 3) * 256 + kc * 128 + (key & 7) * 16) = v;
      fence_proxy_async_smem();
    }
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const bool run = !*abort_flag;

  if (warp >= 8 && warp < 12) {
    regs_dec<kBwdRegsCtl>();
    if (warp == 8 && lane == 0 && run) {
      // ---------------------------------------------------------- producer
      int issued_q[2] = {-1, -1}, issued_d[2] = {-1, -1};
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      tma_prefetch_desc(&tdo);
      mbar_expect_tx(&bars[C_KV], 2 * kTileBytes);
      for (int hf = 0; hf < 2; ++hf) {
        tma_load_3d(big + hf * kHalfTile, &tk, &bars[C_KV], hf * 64, g, row0 + kt * 128);
        tma_load_3d(big + kTileBytes + hf * kHalfTile, &tv, &bars[C_KV], hf * 64, g, row0 + kt * 128);
      }
      int ent = list[0];
#pragma unroll 1
      for (int j = 0; j < n_it; ++j) {
        const int st = j & 1, n = j >> 1;
        const int qt = ent >> 1, h = g * p.G + j % p.G;
        if (j + 1 < n_it) ent = list[(j + 1) / p.G];
        if (qt < kt || qt >= p.NT) {
          *abort_flag = 1;
          atomicOr(p.err, kErrBadList);
          break;
        }
        // Q and dO of a later iteration into L2, so that its load, issued
        // only when a ring stage frees up, finds them there
        if (j + kBwdPrefetch < n_it) {
          const int e2 = list[(j + kBwdPrefetch) / p.G];
          const int qt2 = min(max(e2 >> 1, 0), p.NT - 1), h2 = g * p.G + (j + kBwdPrefetch) % p.G;
          for (int hf = 0; hf < 2; ++hf) {
            tma_prefetch_l2_3d(&tq, hf * 64, h2, row0 + qt2 * 128);
            tma_prefetch_l2_3d(&tdo, hf * 64, h2, row0 + qt2 * 128);
          }
        }
        // Q (and the per-query vectors) of j: the stage frees once dK(j-2) is done
        if (j >= 2 && !mbar_wait(&bars[C_QE + st], (n - 1) & 1, abort_flag, p.err)) break;
        const size_t bt = (((size_t)r * p.Hq + h) * p.NT + qt) * kBiasTileBytes;
        mbar_expect_tx(&bars[C_QF + st], kTileBytes + (uint32_t)kBiasTileBytes);
        bulk_load(bias + st * kBiasTileBytes, p.sbias + bt, (uint32_t)kBiasTileBytes, &bars[C_QF + st]);
        for (int hf = 0; hf < 2; ++hf)
          tma_load_3d(big + (2 + st) * kTileBytes + hf * kHalfTile, &tq, &bars[C_QF + st], hf * 64, h,
                      row0 + qt * 128);
        issued_q[st] = n;
        // dO of j: the stage frees once dV(j-2) is done
        if (j >= 2 && !mbar_wait(&bars[C_DE + st], (n - 1) & 1, abort_flag, p.err)) break;
        mbar_expect_tx(&bars[C_DF + st], kTileBytes + (uint32_t)kBiasTileBytes);
        bulk_load(bias + (2 + st) * kBiasTileBytes, p.dbias + bt, (uint32_t)kBiasTileBytes, &bars[C_DF + st]);
        for (int hf = 0; hf < 2; ++hf)
          tma_load_3d(big + (4 + st) * kTileBytes + hf * kHalfTile, &tdo, &bars[C_DF + st], hf * 64, h,
                      row0 + qt * 128);
        issued_d[st] = n;
      }
      mbar_wait_drain(&bars[C_KV], 0);
      for (int st = 0; st < 2; ++st) {
        if (issued_q[st] >= 0) mbar_wait_drain(&bars[C_QF + st], issued_q[st] & 1);
        if (issued_d[st] >= 0) mbar_wait_drain(&bars[C_DF + st], issued_d[st] & 1);
      }
    } else if (warp == 9 && lane == 0 && run) {
      // ---------------------------------------------------------- MMA issue
      constexpr uint32_t id_kk = idesc_bf16(128, 128, 0, 0);  // S^T, dP^T
      constexpr uint32_t id_kn = idesc_bf16(128, 128, 0, 1);  // dV, dK (A in TMEM)
      // descriptor low words; slice kk adds a constant to the start-address field
      const uint32_t k_km = desc_lo_kmajor(k_s), v_km = desc_lo_kmajor(v_s);
      const uint32_t q_km0 = desc_lo_kmajor(big_s + 2 * kTileBytes), do_km0 = desc_lo_kmajor(big_s + 4 * kTileBytes);
      const uint32_t q_mn0 = desc_lo_mnmajor(big_s + 2 * kTileBytes), do_mn0 = desc_lo_mnmajor(big_s + 4 * kTileBytes);
      constexpr uint32_t kStage = kTileBytes >> 4;  // one tile further in the ring
      auto km = [](int kk) { return (uint32_t)((kk >> 2) * (kHalfTile >> 4) + (kk & 3) * 2); };
      auto mn = [](int kk) { return (uint32_t)(kk * 128); };
      // packed P^T columns of query columns 16 kk .. 16 kk + 15 (dS^T: 32 further)
      auto pk = [](int kk) { return (uint32_t)(128 + (kk >> 2) * 64 + (kk & 3) * 8); };
      const uint32_t bias_s = smem_u32(bias);
      const uint64_t ones = bias_desc(bias_s + 4 * (uint32_t)kBiasTileBytes);
      auto issue_s = [&](int jj) {  // S^T(jj) = K Q(jj)^T, plus -LSE / scale per query
        const uint32_t so = (jj & 1) ? kStage : 0;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ss_lo(tmem, k_km + km(kk), q_km0 + so + km(kk), id_kk, kk > 0);
        mma_ss(tmem, ones, bias_desc(bias_s + (jj & 1) * (uint32_t)kBiasTileBytes), id_kk, 1);
        mma_commit(&bars[C_SF]);
      };
      auto issue_dp = [&](int jj) {  // dP^T(jj) = V dO(jj)^T, minus Delta per query
        const uint32_t so = (jj & 1) ? kStage : 0;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) mma_ss_lo(tmem + 128, v_km + km(kk), do_km0 + so + km(kk), id_kk, kk > 0);
        mma_ss(tmem + 128, ones, bias_desc(bias_s + (2 + (jj & 1)) * (uint32_t)kBiasTileBytes), id_kk, 1);
        mma_commit(&bars[C_DPF]);
      };
      bool ok = mbar_wait(&bars[C_KV], 0, abort_flag, p.err) && mbar_wait(&bars[C_QF], 0, abort_flag, p.err);
      if (ok) {
        fence_after_sync();
        issue_s(0);
        ok = mbar_wait(&bars[C_DF], 0, abort_flag, p.err);
      }
      if (ok) {
        fence_after_sync();
        issue_dp(0);
      }
      // S^T(1) once the pass of 0 has loaded S^T(0)
      if (ok && n_it > 1) {
        ok = mbar_wait(&bars[C_SR], 0, abort_flag, p.err) && mbar_wait(&bars[C_QF + 1], 0, abort_flag, p.err);
        if (ok) {
          fence_after_sync();
          issue_s(1);
        }
      }
#pragma unroll 1
      for (int j = 0; ok && j < n_it; ++j) {
        const int st = j & 1;
        const uint32_t so = st ? kStage : 0;
        if (!mbar_wait(&bars[C_DR], j & 1, abort_flag, p.err)) break;
        fence_after_sync();
        // dK += dS^T Q and dV += P^T dO, both read from the dP^T columns
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts_lo(tmem + 384, tmem + pk(kk) + 32, q_mn0 + so + mn(kk), id_kn, (j > 0 || kk > 0));
        mma_commit(&bars[C_QE + st]);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts_lo(tmem + 256, tmem + pk(kk), do_mn0 + so + mn(kk), id_kn, (j > 0 || kk > 0));
        mma_commit(&bars[C_DE + st]);
        // dP^T(j+1) over them, once the store warps hold dS^T(j)
        if (j + 1 < n_it) {
          if (!mbar_wait(&bars[C_DSR], j & 1, abort_flag, p.err) ||
              !mbar_wait(&bars[C_DF + ((j + 1) & 1)], ((j + 1) >> 1) & 1, abort_flag, p.err))
            break;
          fence_after_sync();
          issue_dp(j + 1);
        }
        // S^T(j+2) once the pass of j+1 has loaded S^T(j+1)
        if (j + 2 < n_it) {
          if (!mbar_wait(&bars[C_SR], (j + 1) & 1, abort_flag, p.err) ||
              !mbar_wait(&bars[C_QF + st], ((j + 2) >> 1) & 1, abort_flag, p.err))
            break;
          fence_after_sync();
          issue_s(j + 2);
        }
      }
      if (ok) mma_commit(&bars[C_DONE]);
      mma_commit(&bars[C_DRAIN]);
      mbar_wait_drain(&bars[C_DRAIN], 0);
    }
    __syncwarp();
  } else if (warp >= 12) {
    // ------------------------------------------------ dS^T store (warps 12-15)
    regs_dec<kBwdRegsStore>();
    const int t = threadIdx.x & 127;     // key row = TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    bool ok = run;
    for (int j = 0; ok && j < n_it; ++j) {
      if (!__all_sync(0xffffffffu, mbar_wait(&bars[C_DR], j & 1, abort_flag, p.err))) break;
      fence_after_sync();
      const int pr_j = pairs[j / p.G];
      uint32_t d0[32], d1[32];           // dS^T of query columns 0..63 and 64..127
      tmem_ld32(tmem + lane_base + 128 + 32, d0);
      tmem_ld32(tmem + lane_base + 192 + 32, d1);
      tmem_ld_wait();
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[C_DSR]);
      if (pr_j >= 0 && pr_j < p.cap) {
        uint8_t* tile = p.ds + ((size_t)pr_j * p.slot_heads + gl * p.G + j % p.G) * kDsTileBytes + t * 16;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          *reinterpret_cast<uint4*>(tile + c * kDsBlock) = make_uint4(d0[4 * c], d0[4 * c + 1], d0[4 * c + 2], d0[4 * c + 3]);
          *reinterpret_cast<uint4*>(tile + (8 + c) * kDsBlock) =
              make_uint4(d1[4 * c], d1[4 * c + 1], d1[4 * c + 2], d1[4 * c + 3]);
        }
      } else if (lane == 0) {
        atomicOr(p.err, kErrCapacity);
      }
    }
  } else {
    // ------------------------------------------------ per-key elementwise
    regs_inc<kBwdRegsMath>();
    const int half = warp >> 2;          // query columns 64 half .. 64 half + 63
    const int t = threadIdx.x & 127;     // key row = TMEM lane
    const int jk = kt * 128 + t;         // key index in the row
    const int se_j = p.se[(size_t)row0 + jk];
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t s_col = lane_base + half * 64, dp_col = lane_base + 128 + half * 64;
    const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
    bool ok = run;
    int ent = run ? list[0] : 0;
    for (int j = 0; ok && j < n_it; ++j) {
      const int qt = ent >> 1, part = ent & 1;
      if (j + 1 < n_it) ent = list[(j + 1) / p.G];
      const int q0 = qt * 128 + half * 64;
      if (!__all_sync(0xffffffffu, mbar_wait(&bars[C_SF], j & 1, abort_flag, p.err))) {
        ok = false;
        break;
      }
      fence_after_sync();
      // P from S^T: 64 query columns of this half; the S^T columns are free
      // for S^T(j+2) once loaded
      uint32_t u[64];
      tmem_ld32(tmem + s_col, u);
      tmem_ld32(tmem + s_col + 32, u + 32);
      tmem_ld_wait();
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[C_SR]);
#pragma unroll
      for (int col = 0; col < 64; col += 4) {
#pragma unroll
        for (int u2 = 0; u2 < 2; ++u2) {
          const int cc = col + 2 * u2;
          float2 y = __fmul2_rn(make_float2(__uint_as_float(u[cc]), __uint_as_float(u[cc + 1])), sl2);
          if (part) {
            const int i = q0 + cc;
            if (!(jk <= i && se_j >= i)) y.x = -INFINITY;
            if (!(jk <= i + 1 && se_j >= i + 1)) y.y = -INFINITY;
          }
          u[cc] = __float_as_uint(ex2(y.x));
          u[cc + 1] = __float_as_uint(ex2(y.y));
        }
      }
      // dS = P (dP - Delta) once dP^T(j) is in TMEM
      if (!__all_sync(0xffffffffu, mbar_wait(&bars[C_DPF], j & 1, abort_flag, p.err))) {
        ok = false;
        break;
      }
      fence_after_sync();
      uint32_t ud[64];
      tmem_ld32(tmem + dp_col, ud);
      tmem_ld32(tmem + dp_col + 32, ud + 32);
      tmem_ld_wait();
      uint32_t pp[32], dd[32];           // P and dS of the 64 columns, packed bf16 pairs
#pragma unroll
      for (int col = 0; col < 64; col += 4) {
#pragma unroll
        for (int u2 = 0; u2 < 2; ++u2) {
          const int cc = col + 2 * u2;
          const float2 pr = make_float2(__uint_as_float(u[cc]), __uint_as_float(u[cc + 1]));
          const float2 ds = __fmul2_rn(pr, make_float2(__uint_as_float(ud[cc]), __uint_as_float(ud[cc + 1])));
          pp[cc >> 1] = pack_bf16x2(pr.x, pr.y);
          dd[cc >> 1] = pack_bf16x2(ds.x, ds.y);
        }
      }
      // P^T and dS^T over the dP^T columns just read
      tmem_st32(tmem + dp_col, pp);
      tmem_st32(tmem + dp_col + 32, dd);
      tmem_st_wait();
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[C_DR]);
    }
    if (ok && mbar_wait(&bars[C_DONE], 0, abort_flag, p.err)) {
      fence_after_sync();
      // warps 0-3 write dV, warps 4-7 dK (times scale)
      const bool is_dv = half == 0;
      __nv_bfloat16* dst = (is_dv ? p.dv : p.dk) + (((size_t)row0 + jk) * p.Hkv + g) * 128;
      const float sc = is_dv ? 1.f : p.scale;
      const uint32_t col0 = lane_base + (is_dv ? 256 : 384);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t u[32];
        tmem_ld32(tmem + col0 + c * 32, u);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint4 a;
          a.x = pack_bf16x2(__uint_as_float(u[8 * k + 0]) * sc, __uint_as_float(u[8 * k + 1]) * sc);
          a.y = pack_bf16x2(__uint_as_float(u[8 * k + 2]) * sc, __uint_as_float(u[8 * k + 3]) * sc);
          a.z = pack_bf16x2(__uint_as_float(u[8 * k + 4]) * sc, __uint_as_float(u[8 * k + 5]) * sc);
          a.w = pack_bf16x2(__uint_as_float(u[8 * k + 6]) * sc, __uint_as_float(u[8 * k + 7]) * sc);
          *reinterpret_cast<uint4*>(dst + c * 32 + 8 * k) = a;
        }
      }
    }
  }

  __syncwarp();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == 9) tmem_dealloc(tmem, 512);
}

struct DqParams {
  int R, T, Hq, Hkv, NT, G, nquad;
  int g0, ng;           // kv heads [g0, g0 + ng) of this launch
  int slot_heads;       // query heads per pair in a dS slot
  int64_t cap;          // dS pairs per slot
  const int32_t* csr_cnt;
  const int32_t* csr;
  const int32_t* csr_off;
  const int32_t* row_base;
  const uint8_t* ds;    // this launch's slot: [pair][slot_heads] dS^T tiles
  __nv_bfloat16* dq;
  float scale;
  uint32_t* err;
};

// No-swizzle shared-memory descriptor of a dS^T tile used as the MN-major A
// operand of the dQ product (M = queries, K = keys): 8 x 16-byte core
// matrices, 2048 bytes apart along M (stride-dimension offset) and 128 bytes
// apart along K (leading-dimension offset).
__device__ __forceinline__ uint64_t ds_desc(uint32_t addr) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(128u >> 4) << 16) |
         ((uint64_t)(uint32_t(kDsBlock) >> 4) << 32) | (1ull << 46);
}

enum { Q_KF = 0, Q_KE = 2, Q_DF = 4, Q_DE = 8, Q_DONE = 12, Q_DRAIN = 13, Q_COUNT = 14 };
// shared memory: [K0 | K1 | dS0 .. dS3] (1024-aligned) [barriers ...]
constexpr int kDqBigBytes = 6 * kTileBytes;
constexpr int kDqSmem = kDqBigBytes + kSmallBytes;
static_assert(kDqSmem <= kSmemLimit, "dQ shared memory");
constexpr int kDqThreads = 256;  // warp 0 loads, warp 1 MMA, warps 4-7 write dQ

__global__ void __launch_bounds__(kDqThreads, 1)
    dq_tc_kernel(const __grid_constant__ CUtensorMap tk, const DqParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* big = smem_raw;
  const uint32_t big_s = smem_u32(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw + kDqBigBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Q_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // longest lists (highest query tiles) first
  const int per_qt = p.R * p.ng * p.nquad;
  const int qt = p.NT - 1 - (int)(blockIdx.x / per_qt);
  int rem = blockIdx.x % per_qt;
  const int r = rem / (p.ng * p.nquad);
  rem %= p.ng * p.nquad;
  const int gl = rem / p.nquad, quad = rem % p.nquad;  // kv head within this launch
  const int g = p.g0 + gl;
  const int h0 = g * p.G + 4 * quad;
  const int nh = min(4, p.G - 4 * quad);
  const int cnt = p.csr_cnt[(size_t)r * p.NT + qt];
  const int32_t* list = p.csr + ((size_t)r * p.NT + qt) * p.NT;
  const int64_t pbase = (int64_t)p.row_base[r] + p.csr_off[(size_t)r * p.NT + qt];
  const int row0 = r * p.T;

  if (threadIdx.x == 0) {
    for (int b = 0; b < Q_COUNT; ++b) mbar_init(&bars[b], 1);
    *abort_flag = 0;
    if ((big_s & 1023u) != 0 || cnt <= 0 || cnt > p.NT) {
      *abort_flag = 1;
      atomicOr(p.err, (big_s & 1023u) != 0 ? kErrTmem : kErrBadList);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const bool run = !*abort_flag;

  if (warp == 0 && lane == 0 && run) {
    // ------------------------------------------------------------ loads
    tma_prefetch_desc(&tk);
    int issued_k[2] = {-1, -1}, issued_d[4] = {-1, -1, -1, -1};
    int d = 0;
    for (int e = 0; e < cnt; ++e) {
      const int kt = list[e] >> 1, sk = e & 1;
      const int64_t pair = pbase + e;
      if (kt > qt || pair >= p.cap) {
        *abort_flag = 1;
        atomicOr(p.err, kt > qt ? kErrBadList : kErrCapacity);
        break;
      }
      if (e >= 2 && !mbar_wait(&bars[Q_KE + sk], ((e >> 1) - 1) & 1, abort_flag, p.err)) break;
      mbar_expect_tx(&bars[Q_KF + sk], kTileBytes);
      for (int hf = 0; hf < 2; ++hf)
        tma_load_3d(big + sk * kTileBytes + hf * kHalfTile, &tk, &bars[Q_KF + sk], hf * 64, g, row0 + kt * 128);
      issued_k[sk] = e >> 1;
      bool ok = true;
      for (int hh = 0; hh < nh; ++hh, ++d) {
        const int sd = d & 3;
        if (d >= 4 && !mbar_wait(&bars[Q_DE + sd], ((d >> 2) - 1) & 1, abort_flag, p.err)) {
          ok = false;
          break;
        }
        mbar_expect_tx(&bars[Q_DF + sd], (uint32_t)kDsTileBytes);
        bulk_load(big + (2 + sd) * kTileBytes,
                  p.ds + ((size_t)pair * p.slot_heads + gl * p.G + 4 * quad + hh) * kDsTileBytes,
                  (uint32_t)kDsTileBytes, &bars[Q_DF + sd]);
        issued_d[sd] = d >> 2;
      }
      if (!ok) break;
    }
    for (int s = 0; s < 2; ++s)
      if (issued_k[s] >= 0) mbar_wait_drain(&bars[Q_KF + s], issued_k[s] & 1);
    for (int s = 0; s < 4; ++s)
      if (issued_d[s] >= 0) mbar_wait_drain(&bars[Q_DF + s], issued_d[s] & 1);
  } else if (warp == 1 && lane == 0 && run) {
    // ------------------------------------------------------------ MMA
    constexpr uint32_t id_nn = idesc_bf16(128, 128, 1, 1);  // A = dS (queries contiguous), B = K
    auto mn = [](int kk) { return (uint32_t)(kk * 128); };
    bool ok = true;
    int d = 0;
    for (int e = 0; ok && e < cnt; ++e) {
      const int sk = e & 1;
      if (!mbar_wait(&bars[Q_KF + sk], (e >> 1) & 1, abort_flag, p.err)) {
        ok = false;
        break;
      }
      const uint32_t k_mn = desc_lo_mnmajor(big_s + sk * kTileBytes);
      for (int hh = 0; hh < nh; ++hh, ++d) {
        const int sd = d & 3;
        if (!mbar_wait(&bars[Q_DF + sd], (d >> 2) & 1, abort_flag, p.err)) {
          ok = false;
          break;
        }
        fence_after_sync();
        // slice kk = keys 16 kk .. 16 kk + 15: two core matrices along K, 256 bytes further
        const uint64_t ds_a = ds_desc(big_s + (2 + sd) * kTileBytes);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss_a64(tmem + hh * 128, ds_a + (uint64_t)(kk * 16), k_mn + mn(kk), id_nn, (e > 0 || kk > 0));
        mma_commit(&bars[Q_DE + sd]);
      }
      if (ok) mma_commit(&bars[Q_KE + sk]);
    }
    if (ok) mma_commit(&bars[Q_DONE]);
    mma_commit(&bars[Q_DRAIN]);
    mbar_wait_drain(&bars[Q_DRAIN], 0);
  } else if (warp >= 4 && run) {
    // ------------------------------------------------------------ dQ out
    const int t = threadIdx.x - 128;   // query row = TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    if (mbar_wait(&bars[Q_DONE], 0, abort_flag, p.err)) {
      fence_after_sync();
      for (int hh = 0; hh < nh; ++hh) {
        __nv_bfloat16* out = p.dq + (((size_t)row0 + qt * 128 + t) * p.Hq + h0 + hh) * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t u[32];
          tmem_ld32(tmem + lane_base + hh * 128 + c * 32, u);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint4 a;
            a.x = pack_bf16x2(__uint_as_float(u[8 * k + 0]) * p.scale, __uint_as_float(u[8 * k + 1]) * p.scale);
            a.y = pack_bf16x2(__uint_as_float(u[8 * k + 2]) * p.scale, __uint_as_float(u[8 * k + 3]) * p.scale);
            a.z = pack_bf16x2(__uint_as_float(u[8 * k + 4]) * p.scale, __uint_as_float(u[8 * k + 5]) * p.scale);
            a.w = pack_bf16x2(__uint_as_float(u[8 * k + 6]) * p.scale, __uint_as_float(u[8 * k + 7]) * p.scale);
            *reinterpret_cast<uint4*>(out + c * 32 + 8 * k) = a;
          }
        }
      }
    }
  }

  __syncwarp();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// Delta[r,h,i] = sum_d dO . O (bf16 in, f32) for every (row, token, head);
// writes the two bias tiles of the token's query tile: -LSE_i / scale and
// -Delta_i, each as three bf16 terms (hi, mid, lo: hi = bf16(x), mid =
// bf16(x - hi), lo = bf16(x - hi - mid)) in columns 0-2 of the query's row,
// zeros elsewhere (layout of bias_desc).
__device__ __forceinline__ uint4 bias_row(float x) {
  const __nv_bfloat16 hi = __float2bfloat16_rn(x);
  const float r1 = x - __bfloat162float(hi);
  const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
  const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
  return make_uint4((uint32_t)__bfloat16_as_ushort(hi) | ((uint32_t)__bfloat16_as_ushort(mid) << 16),
                    (uint32_t)__bfloat16_as_ushort(lo), 0u, 0u);
}

__global__ void __launch_bounds__(256) bwd_delta_kernel(const __nv_bfloat16* __restrict__ o,
                                                        const __nv_bfloat16* __restrict__ dout,
                                                        const float* __restrict__ lse,
                                                        uint8_t* __restrict__ sbias,
                                                        uint8_t* __restrict__ dbias, float inv_scale, int R,
                                                        int T, int Hq) {
  // 16 lanes per (token, head) row of 128 values, 16 bytes of O and of dO per
  // lane; each half-warp takes kRowsPer rows per pass with all their loads
  // issued first, so that enough bytes are in flight to stream O and dO
  constexpr int kRowsPer = 4;
  const int hl = threadIdx.x & 15;
  const unsigned hmask = 0xffffu << (threadIdx.x & 16);   // the half-warps loop independently
  const size_t rows = (size_t)R * T * Hq;
  const int NT = T / 128;
  const size_t n_half = (size_t)gridDim.x * (blockDim.x / 16);
  for (size_t w0 = ((size_t)blockIdx.x * (blockDim.x / 16) + (threadIdx.x >> 4)) * kRowsPer; w0 < rows;
       w0 += n_half * kRowsPer) {
    uint4 a[kRowsPer], b[kRowsPer];
#pragma unroll
    for (int k = 0; k < kRowsPer; ++k) {
      const size_t w = w0 + k;
      a[k] = b[k] = make_uint4(0, 0, 0, 0);
      if (w < rows) {
        a[k] = reinterpret_cast<const uint4*>(o + w * 128)[hl];
        b[k] = reinterpret_cast<const uint4*>(dout + w * 128)[hl];
      }
    }
#pragma unroll
    for (int k = 0; k < kRowsPer; ++k) {
      const size_t w = w0 + k;
      const uint32_t wa[4] = {a[k].x, a[k].y, a[k].z, a[k].w}, wb[4] = {b[k].x, b[k].y, b[k].z, b[k].w};
      float acc = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc = fmaf(__uint_as_float(wa[q] << 16), __uint_as_float(wb[q] << 16), acc);
        acc = fmaf(__uint_as_float(wa[q] & 0xffff0000u), __uint_as_float(wb[q] & 0xffff0000u), acc);
      }
#pragma unroll
      for (int sft = 8; sft > 0; sft >>= 1) acc += __shfl_xor_sync(hmask, acc, sft);
      if (w < rows && hl < 2) {
        const int h = (int)(w % Hq);
        const size_t ri = w / Hq;
        const size_t rr = ri / T, i = ri - rr * T;
        const size_t tile = ((rr * Hq + h) * NT + i / 128) * kBiasTileBytes;
        const int q = (int)(i & 127);
        const size_t at = tile + (q >> 3) * 256 + (q & 7) * 16;
        uint8_t* dst = hl == 0 ? sbias : dbias;
        const float x = hl == 0 ? -lse[(rr * Hq + h) * T + i] * inv_scale : -acc;
        *reinterpret_cast<uint4*>(dst + at) = bias_row(x);
        *reinterpret_cast<uint4*>(dst + at + 128) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }
}

}  // namespace

cudaError_t tc_fwd(const AttnArgs& a, cudaStream_t s) {
  CUtensorMap mq, mk, mv;
  const int64_t rows = (int64_t)a.R * a.T;
  if (!make_map(&mq, a.q, rows, a.Hq) || !make_map(&mk, a.k, rows, a.Hkv) ||
      !make_map(&mv, a.v, rows, a.Hkv))
    return cudaErrorInvalidValue;
  FwdParams p;
  p.R = a.R;
  p.T = a.T;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.NT = a.T / 128;
  p.G = a.Hq / a.Hkv;
  p.npairs = (p.G + 1) / 2;
  p.scale_log2 = a.scale * kLog2e;
  p.se = a.se;
  p.csr_cnt = a.csr_cnt;
  p.csr = a.csr;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.lse = a.lse;
  p.err = a.err;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemLimit);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const unsigned grid = (unsigned)(p.NT * p.R * p.Hkv * p.npairs);
  fwd_tc_kernel<<<grid, kThreads, kSmemLimit, s>>>(mq, mk, mv, p);
  return cudaGetLastError();
}


}  // namespace stp

namespace stp {

namespace {

// Library-owned streams of the backward's kv-head groups: a pool per device,
// created on first use, handed out round-robin so that backward calls made
// from different caller streams do not serialize on the same ones.  Every
// enqueue sequence that uses the pool holds g_bwd_mu.
constexpr int kBwdPool = 16;
struct BwdStreams {
  bool ready = false;
  int next = 0;
  cudaStream_t s[kBwdPool] = {};
  cudaEvent_t fork = nullptr, join[kBwdPool] = {};
};
std::mutex g_bwd_mu;
BwdStreams g_bwd_streams[64];

cudaError_t bwd_streams(BwdStreams** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  BwdStreams& b = g_bwd_streams[dev];
  if (!b.ready) {
    e = cudaEventCreateWithFlags(&b.fork, cudaEventDisableTiming);
    for (int i = 0; i < kBwdPool && e == cudaSuccess; ++i) {
      e = cudaStreamCreateWithFlags(&b.s[i], cudaStreamNonBlocking);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&b.join[i], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) return e;
    b.ready = true;
  }
  *out = &b;
  return cudaSuccess;
}

}  // namespace

cudaError_t tc_bwd(const AttnArgs& a, cudaStream_t s) {
  CUtensorMap mq, mk, mv, mdo;
  const int64_t rows = (int64_t)a.R * a.T;
  if (!make_map(&mq, a.q, rows, a.Hq) || !make_map(&mk, a.k, rows, a.Hkv) ||
      !make_map(&mv, a.v, rows, a.Hkv) || !make_map(&mdo, a.dout, rows, a.Hq))
    return cudaErrorInvalidValue;
  bwd_delta_kernel<<<2048, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(a.o_in),
                                        static_cast<const __nv_bfloat16*>(a.dout), a.lse,
                                        static_cast<uint8_t*>(a.sbias), static_cast<uint8_t*>(a.dbias),
                                        1.f / a.scale, a.R, a.T, a.Hq);
  const BwdGroups grp = bwd_groups(a.Hq, a.Hkv, a.ds_slots);
  BwdParams p;
  p.R = a.R;
  p.T = a.T;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.NT = a.T / 128;
  p.G = a.Hq / a.Hkv;
  p.slot_heads = grp.group_heads;
  p.scale_log2 = a.scale * kLog2e;
  p.scale = a.scale;
  p.cap = a.ds_cap;
  p.se = a.se;
  p.csc_cnt = a.csc_cnt;
  p.csc = a.csc;
  p.csc_pair = a.csc_pair;
  p.sbias = static_cast<const uint8_t*>(a.sbias);
  p.dbias = static_cast<const uint8_t*>(a.dbias);
  p.dk = static_cast<__nv_bfloat16*>(a.dk);
  p.dv = static_cast<__nv_bfloat16*>(a.dv);
  p.err = a.err;
  DqParams q;
  q.R = a.R;
  q.T = a.T;
  q.Hq = a.Hq;
  q.Hkv = a.Hkv;
  q.NT = p.NT;
  q.G = p.G;
  q.nquad = (p.G + 3) / 4;
  q.slot_heads = grp.group_heads;
  q.cap = a.ds_cap;
  q.csr_cnt = a.csr_cnt;
  q.csr = a.csr;
  q.csr_off = a.csr_off;
  q.row_base = a.row_base;
  q.dq = static_cast<__nv_bfloat16*>(a.dq);
  q.scale = a.scale;
  q.err = a.err;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kBwdSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(dq_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDqSmem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  // The kv heads in grp.n groups, each on its own stream: a group's dQ pass
  // (HBM-bound) starts as soon as that group's dK/dV kernel is done and runs
  // while the other groups compute.  Group gi keeps its dS tiles in slot
  // gi % slots; when slots < groups, it first waits for the dQ pass of group
  // gi - slots, the slot's previous user.
  const int n_groups = grp.n, slots = grp.slots;
  std::lock_guard<std::mutex> lock(g_bwd_mu);
  BwdStreams* bs = nullptr;
  if (n_groups > 1) {
    cudaError_t e = bwd_streams(&bs);
    if (e != cudaSuccess) return e;
    e = cudaEventRecord(bs->fork, s);
    if (e != cudaSuccess) return e;
  }
  int stream_of[kBwdGroups] = {};
  for (int gi = 0; gi < n_groups; ++gi) {
    const int g0 = gi * p.Hkv / n_groups, g1 = (gi + 1) * p.Hkv / n_groups;
    cudaStream_t sg = s;
    const int slot = n_groups > 1 ? (bs->next + gi) % kBwdPool : 0;
    stream_of[gi] = slot;
    if (n_groups > 1) {
      sg = bs->s[slot];
      cudaError_t e = cudaStreamWaitEvent(sg, bs->fork, 0);
      if (e == cudaSuccess && gi >= slots) e = cudaStreamWaitEvent(sg, bs->join[stream_of[gi - slots]], 0);
      if (e != cudaSuccess) return e;
    }
    p.g0 = q.g0 = g0;
    p.ng = q.ng = g1 - g0;
    p.ds = static_cast<uint8_t*>(a.ds) + (size_t)(gi % slots) * a.ds_slot_bytes;
    q.ds = p.ds;
    bwd_tc_kernel<<<(unsigned)(p.NT * p.R * p.ng), kBwdThreads, kBwdSmem, sg>>>(mq, mk, mv, mdo, p);
    dq_tc_kernel<<<(unsigned)(p.NT * p.R * q.ng * q.nquad), kDqThreads, kDqSmem, sg>>>(mk, q);
    if (n_groups > 1) {
      cudaError_t e = cudaEventRecord(bs->join[slot], sg);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(s, bs->join[slot], 0);
      if (e != cudaSuccess) return e;
    }
  }
  if (n_groups > 1) bs->next = (bs->next + n_groups) % kBwdPool;
  return cudaGetLastError();
}

}  // namespace stp
