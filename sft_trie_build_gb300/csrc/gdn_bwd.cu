// Tree-aware Gated DeltaNet layer core, backward ("Prefix tree packing", GDN
// section: a child's initial state is its parent's final state, so the
// parent's final-state gradient is the sum of its children's initial-state
// gradients; roots start from zero).  For L = sum dO . o, per head and per
// chunk of n tokens (S0 its starting state, saved by the training forward,
// gam = cumsum(g) inside the chunk, the chunk's operands from the forward):
//   walk:   dV' = P^T dO + K~ dS_n,   dS0 = Q~^T dO + e^{gam_n} dS_n - W^T dV'
//   chunk:  dQ~ = dO S0^T, dP = dO V'^T, dK~ = V' dS_n^T, dW = -dV' S0^T, dU^ = dV',
//           dT = dU^ (beta V)^T + dW (beta e^gam K)^T, dA = -lower(T^T dT T^T)
//           (T = (I + A)^{-1}), then through Q~, K~, P, A, U^ and W to dq, dk,
//           dv, dbeta and dgam, and dg = the reverse cumulative sum of dgam
//   tokens: through the unit-norm q, k heads, SiLU and the path convolution.
// Five kernels:
//   gdn_bwd_walk_kernel   one launch per depth, deepest first; one CTA per
//                         (segment, head) walks its chunks last to first with
//                         the state gradient in TMEM, starting from the sum
//                         of its children's start gradients; both products
//                         per chunk on the tensor core (tcgen05).
//   gdn_bwd_chunk_kernel  one CTA per (chunk, head): everything above that
//                         needs only the chunk and its two state (gradient)s,
//                         its contractions on the tensor core (tcgen05).
//   gdn_bwd_token_kernel  one block per (64 tokens, q / k / v head): back
//                         through the unit-norm heads and SiLU to dz, the
//                         gradient of the convolution's output (in place of
//                         dy), and the block's share of the weight gradient;
//   gdn_bwd_dx_kernel     the convolution's input gradient of each token,
//                         gathered from the tokens that read it: itself, its
//                         path successors and theirs, three steps down (the
//                         plan's successor lists), in a fixed order;
//   gdn_bwd_dw_kernel     the weight gradient: the blocks' shares summed in
//                         block order.
// No float atomics: every output is summed in one fixed order.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "gdn_common.h"
#include "internal.h"
#include "layout.h"
#include "tc_ptx.cuh"

namespace stp {
namespace {

using namespace tc;

constexpr int kD = kGdnD, kC = kGdnChunk;
constexpr int kBT = 256;   // threads of every backward kernel

struct GbParams {
  int N, H, C, seg0, chunk0;   // seg0, chunk0: first segment / chunk of a launch
  float scale;
  const int32_t* prev;
  const int32_t* prev2;
  const int32_t* prev3;
  const int32_t* seg_len;
  const int32_t* seg_chunk0;
  const int32_t* child_off;
  const int32_t* child;
  const int32_t* chunk_start;
  const int32_t* chunk_len;
  const __nv_bfloat16* x;    // [N, C]
  const float* conv_w;       // [C, 4]
  const float* g;            // [N, H]
  const float* beta;         // [N, H]
  const float* d_o;          // [N, H, d]
  const __nv_bfloat16* y;    // [N, C] conv output (q^, k^ unit heads; v)
  const __nv_bfloat16* wq;   // [rows 128, d]  rows 0-63 Q~, 64-127 W
  const __nv_bfloat16* kt;   // [rows 64, d]
  const __nv_bfloat16* pm;   // [rows 64, 64]
  const float* ut;           // [rows, d, 64]
  const float* decay;        // [rows]
  const float* s0;           // [rows, d_v, d_k]
  float* dsend;              // [rows, d, d]
  float* dvp;                // [rows, 64, d]
  float* sgrad;              // [n_seg H, d, d]
  float* dqkv;               // [N, C]
  float* dwp;                // [N / 64 blocks, C, 4] weight-gradient shares
  const int32_t* succ_off;   // [N + 1] successor lists (CSR) of every token
  const int32_t* succ;
  float* dx;                 // [N, C]
  float* dconv_w;            // [C, 4]
  float* dg;                 // [N, H]
  float* dbeta;              // [N, H]
  uint32_t* err;             // device error word of the workspace
};

typedef CUresult (*EncodeFnB)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFnB encode_bwd() {
  static EncodeFnB fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* q = nullptr;
    cudaDriverEntryPointQueryResult r;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &q, 12000, cudaEnableDefault, &r) ==
            cudaSuccess &&
        r == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFnB>(q);
  });
  return fn;
}

// [rows, cols] bf16 as a 2-D tensor; boxes of 64 columns x box_rows rows, 128-byte swizzled.
bool map_2d(CUtensorMap* m, const void* base, int64_t rows, int cols, int box_rows) {
  EncodeFnB enc = encode_bwd();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [rows, cols] of `esize`-byte elements as a 2-D tensor; boxes of 128 columns
// x box_rows rows, no swizzle (rows of 128 elements in shared memory).
bool map_rows(CUtensorMap* m, const void* base, CUtensorMapDataType type, int esize, int64_t rows, int cols,
              int box_rows) {
  EncodeFnB enc = encode_bwd();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * esize};
  cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, type, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

// MN-major 128-byte-swizzled operand whose 64-element halves lie 8 KB apart.
__device__ __forceinline__ uint32_t desc_lo_mn8k(uint32_t addr) {
  return ((addr & 0x3FFFFu) >> 4) | ((8192u >> 4) << 16);
}

// ---------------------------------------------------------------------------
// Reverse walk of one (segment, head) on the tensor core.  The state gradient
// dS [d_k lanes][d_v columns] lives in TMEM (float32, columns 0-127) for the
// whole segment, starting from the sum of the children's start gradients;
// per chunk, last to first:
//   E1  dS (= dS_n of this chunk) goes out (transposed, for the chunk pass),
//       becomes the bf16 operand DSB, and is decayed in place by e^{gam_n};
//       the chunk's dO rows become bf16 rows 0-63 of its DOV buffer (two
//       buffers alternate, so these writes never wait for the products of
//       the chunk before);
//   M1  dV' = P^T dO + K~ dS_n into columns 128-255 (rows = the chunk's
//       tokens; lanes 64-127 see padding rows and are not read);
//   E2  dV' goes out (transposed) and -dV' becomes rows 64-127 of DOV;
//   M2  dS += [Q~^T | W^T] [dO ; -dV']  (the [Q~; W] tile read MN-major).
// The segment's start gradient dS0 goes out at the end.
// kWkEpiWarps epilogue warps (thread = TMEM lane and kWkCw of its columns),
// then a loads warp ([Q~; W], K~, P of the next chunk into the other of two
// stages) and the MMA warp, which owns TMEM.
// Global layouts written here (each warp's stores contiguous): dS_n of a
// chunk and a segment's dS0 as [d_v][d_k], dV' of a chunk as [d_v][64].
constexpr int kWkEpiWarps = 16;                  // epilogue warps: kWkEpiWarps / 4 per TMEM lane group (8 measured slower)
constexpr int kWkCw = 512 / kWkEpiWarps;         // columns of a TMEM lane per epilogue thread
constexpr int kWkThreads = 32 * kWkEpiWarps + 64;   // then a loads warp and an MMA warp
static_assert(kWkCw % 32 == 0 && kWkCw <= 64, "walk kernel column split");
constexpr int kWkStage = 57344;                  // [Q~; W] 32 KB | K~ 16 KB | P 8 KB
constexpr int kWkOffKt = 32768, kWkOffP = 49152;
constexpr int kWkOffDsb = 2 * kWkStage;          // dS_n bf16 [128 d_k][128 d_v], MN-major B
constexpr int kWkOffDov = kWkOffDsb + 32768;     // 2 x [dO ; -dV'] bf16 [128][128], MN-major B
constexpr int kWkOffBar = kWkOffDov + 2 * 32768;
constexpr int kWkSmem = kWkOffBar + 256 + 1024;
enum { W_F = 0, W_E = 2, W_E1 = 4, W_M1 = 5, W_E2 = 6, W_M2 = 7, W_DRAIN = 8, W_COUNT = 9 };

// Writes 8 bf16 (columns 8c .. 8c+7 of row `row`) into a 128-byte-swizzled
// tile of `rows` rows whose two 64-column halves are rows * 128 bytes apart.
__device__ __forceinline__ void st_sw8(uint8_t* tile, int rows, int row, int c, uint4 v) {
  uint8_t* half = tile + (c >> 3) * rows * 128;
  *reinterpret_cast<uint4*>(half + row * 128 + (((c & 7) ^ (row & 7)) << 4)) = v;
}

__device__ __forceinline__ uint4 pack8(const float* f) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

__global__ void __launch_bounds__(kWkThreads, 1)
    gdn_bwd_walk_kernel(const __grid_constant__ CUtensorMap mwq, const __grid_constant__ CUtensorMap mkt,
                        const __grid_constant__ CUtensorMap mpm, const GbParams p) {
  extern __shared__ uint8_t wsm_dyn[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(wsm_dyn) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kWkOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + W_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seg = p.seg0 + (int)(blockIdx.x / p.H), h = (int)(blockIdx.x % p.H);
  const int c0 = p.seg_chunk0[seg], nck = (p.seg_len[seg] + kC - 1) / kC;

  if (threadIdx.x == 0) {
    for (int b = 0; b < W_COUNT; ++b) mbar_init(&bars[b], (b == W_E1 || b == W_E2) ? kWkEpiWarps : 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWkEpiWarps + 1) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == kWkEpiWarps) {
    if (lane == 0) {
      // ------------------------------------------------------------ loads
      tma_prefetch_desc(&mwq);
      tma_prefetch_desc(&mkt);
      tma_prefetch_desc(&mpm);
      int last[2] = {-1, -1};
      for (int n = 0; n < nck; ++n) {   // n-th chunk processed = chunk nck - 1 - n
        const int st = n & 1;
        if (n >= 2 && !mbar_wait(&bars[W_E + st], ((n >> 1) - 1) & 1, abort_flag, p.err)) break;
        const int row = (c0 + nck - 1 - n) * p.H + h;
        uint8_t* stage = sm + st * kWkStage;
        mbar_expect_tx(&bars[W_F + st], 32768 + 16384 + 8192);
        tma_load_2d(stage, &mwq, &bars[W_F + st], 0, row * 128);
        tma_load_2d(stage + 16384, &mwq, &bars[W_F + st], 64, row * 128);
        tma_load_2d(stage + kWkOffKt, &mkt, &bars[W_F + st], 0, row * kC);
        tma_load_2d(stage + kWkOffKt + 8192, &mkt, &bars[W_F + st], 64, row * kC);
        tma_load_2d(stage + kWkOffP, &mpm, &bars[W_F + st], 0, row * kC);
        last[st] = (n >> 1) & 1;
      }
      for (int st = 0; st < 2; ++st)
        if (last[st] >= 0) mbar_wait_drain(&bars[W_F + st], last[st]);
    }
    __syncwarp();
  } else if (warp == kWkEpiWarps + 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA
      constexpr uint32_t id_mnmn = idesc_bf16(128, 128, 1, 1);
      constexpr uint32_t id_kmn = idesc_bf16(128, 128, 0, 1);
      const uint32_t dsb = sb + kWkOffDsb;
      for (int n = 0; n < nck; ++n) {
        const int st = n & 1;
        const uint32_t stage = sb + st * kWkStage, dov = sb + kWkOffDov + st * 32768;
        if (!mbar_wait(&bars[W_F + st], (n >> 1) & 1, abort_flag, p.err)) break;
        if (!mbar_wait(&bars[W_E1], n & 1, abort_flag, p.err)) break;
        fence_after_sync();
        // dV' = P^T dO (A = P read MN-major; its rows are the chunk's tokens) ...
#pragma unroll
        for (int s = 0; s < 4; ++s)
          mma_ss_lo(tmem + 128, desc_lo_mn8k(stage + kWkOffP + s * 2048), desc_lo_mnmajor(dov + s * 2048),
                    id_mnmn, s > 0 ? 1u : 0u);
        // ... + K~ dS_n (A = K~ K-major)
#pragma unroll
        for (int s = 0; s < 8; ++s)
          mma_ss_lo(tmem + 128, desc_lo_kmajor(stage + kWkOffKt + (s >> 2) * 8192 + (s & 3) * 32),
                    desc_lo_mnmajor(dsb + s * 2048), id_kmn, 1u);
        mma_commit(&bars[W_M1]);
        if (!mbar_wait(&bars[W_E2], n & 1, abort_flag, p.err)) break;
        fence_after_sync();
        // dS += [Q~^T | W^T] [dO ; -dV']
#pragma unroll
        for (int s = 0; s < 8; ++s)
          mma_ss_lo(tmem, desc_lo_mnmajor(stage + s * 2048), desc_lo_mnmajor(dov + s * 2048), id_mnmn, 1u);
        mma_commit(&bars[W_M2]);
        mma_commit(&bars[W_E + st]);
      }
      mma_commit(&bars[W_DRAIN]);
      mbar_wait_drain(&bars[W_DRAIN], 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // thread = (TMEM lane r, kWkCw columns from col0): the warps w, w + 4, ...
    // share lanes 32 (w % 4) ..
    const int r = threadIdx.x & 127;   // r: d_k row of dS; token row of dV'
    const uint32_t lrow = (uint32_t)((warp & 3) * 32) << 16, col0 = (uint32_t)(warp >> 2) * kWkCw;
    const int pc0 = (int)col0 >> 3;   // this thread's first 16-byte piece of a bf16 operand row
    uint8_t* dsb = sm + kWkOffDsb;
    uint32_t v[32];
    // dO rows of the n-th chunk processed into DOV buffer n % 2 (rows 0-63),
    // by the threads of the warps w with w % 4 >= 2 (index u): 64 rows x 16
    // pieces of 8 columns, all loads of a thread in flight at once
    constexpr int kNu = 16 * kWkEpiWarps, kPer = 1024 / kNu;
    auto load_do = [&](int n, int u) {
      const int c = c0 + nck - 1 - n, L = p.chunk_len[c], x0 = p.chunk_start[c];
      uint8_t* dov = sm + kWkOffDov + (n & 1) * 32768;
      const float* dO = p.d_o + (size_t)x0 * p.H * kD + h * kD;
      float4 a[kPer], b[kPer];
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int e = u + kNu * k, t = e >> 4, c8 = e & 15;
        a[k] = b[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t < L) {
          const float4* src = reinterpret_cast<const float4*>(dO + (size_t)t * p.H * kD + c8 * 8);
          a[k] = src[0];
          b[k] = src[1];
        }
      }
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int e = u + kNu * k, t = e >> 4, c8 = e & 15;
        const float f[8] = {a[k].x, a[k].y, a[k].z, a[k].w, b[k].x, b[k].y, b[k].z, b[k].w};
        st_sw8(dov, 128, t, c8, pack8(f));
      }
    };
    {   // the segment's end gradient: the sum of its children's start gradients
      const int k0 = p.child_off[seg], k1 = p.child_off[seg + 1];
#pragma unroll 1
      for (int cc = 0; cc < kWkCw / 32; ++cc) {
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          float a = 0.f;
          for (int c = k0; c < k1; ++c)
            a += p.sgrad[(((size_t)p.child[c] * p.H + h) * kD + col0 + cc * 32 + q) * kD + r];
          v[q] = __float_as_uint(a);
        }
        tmem_st32(tmem + lrow + col0 + cc * 32, v);
      }
      tmem_st_wait();
    }
    bool ok = true;
    // The warps w with w % 4 < 2 make -dV' (E2: TMEM lanes 0-63); the others
    // load the dO rows, each chunk's while the chunk before it is finished:
    // the DOV buffer of chunk n + 1 was last read by the products of chunk
    // n - 1, complete before E1 of chunk n.
    const bool e2_warp = (warp & 3) < 2;
    const int u = ((warp >> 2) * 2 + (warp & 1)) * 32 + lane;
    if (nck > 0 && !e2_warp) load_do(0, u);
    for (int n = 0; ok && n < nck; ++n) {
      const int c = c0 + nck - 1 - n;
      const size_t row = (size_t)c * p.H + h;
      const float dec = p.decay[row];
      if (n > 0) {
        if (!__all_sync(0xffffffffu, mbar_wait(&bars[W_M2], (n - 1) & 1, abort_flag, p.err))) {
          ok = false;
          break;
        }
        fence_after_sync();
      }
      // E1: dS_n to the bf16 operand and decayed in place, then (off the
      // chain: the products of this chunk already run) out to global
      // memory ([d_v][d_k]) from registers
      float* dse = p.dsend + row * kD * kD;
      uint32_t vv[kWkCw];
#pragma unroll
      for (int cc = 0; cc < kWkCw / 32; ++cc) tmem_ld32(tmem + lrow + col0 + cc * 32, vv + cc * 32);
      tmem_ld_wait();
#pragma unroll
      for (int cc = 0; cc < kWkCw / 32; ++cc) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          st_sw8(dsb, 128, r, pc0 + cc * 4 + j, pack8(reinterpret_cast<const float*>(vv) + cc * 32 + 8 * j));
      }
      fence_proxy_async_smem();
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[W_E1]);
      // the decayed dS goes back while the first products run (they read the
      // bf16 copy); the second adds to it only after every warp's W_E2 arrival
#pragma unroll
      for (int cc = 0; cc < kWkCw / 32; ++cc) {
#pragma unroll
        for (int q = 0; q < 32; ++q) v[q] = __float_as_uint(__uint_as_float(vv[cc * 32 + q]) * dec);
        tmem_st32(tmem + lrow + col0 + cc * 32, v);
      }
      tmem_st_wait();
      if (!e2_warp) {   // the E2 warps arrive once -dV' is in place too
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[W_E2]);   // this warp's part of dS is stored
      }
#pragma unroll
      for (int q = 0; q < kWkCw; ++q) dse[(col0 + q) * kD + r] = __uint_as_float(vv[q]);
      if (!e2_warp && n + 1 < nck) load_do(n + 1, u);
      // E2: dV' out ([d_v][64]) and -dV' into rows 64-127 of this chunk's DOV
      uint8_t* dov = sm + kWkOffDov + (n & 1) * 32768;
      if (e2_warp) {
        if (!__all_sync(0xffffffffu, mbar_wait(&bars[W_M1], n & 1, abort_flag, p.err))) {
          ok = false;
          break;
        }
        fence_after_sync();
        float* dvo = p.dvp + row * kC * kD;
#pragma unroll
        for (int cc = 0; cc < kWkCw / 32; ++cc) tmem_ld32(tmem + 128 + lrow + col0 + cc * 32, vv + cc * 32);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < kWkCw / 8; ++j) {
          float f[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) f[k] = -__uint_as_float(vv[8 * j + k]);
          st_sw8(dov, 128, kC + r, pc0 + j, pack8(f));
        }
        fence_proxy_async_smem();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[W_E2]);
        // dV' out ([d_v][64]) once the next product may start
#pragma unroll
        for (int q = 0; q < kWkCw; ++q) dvo[(col0 + q) * kC + r] = __uint_as_float(vv[q]);
      }
    }
    if (ok && (nck == 0 || __all_sync(0xffffffffu, mbar_wait(&bars[W_M2], (nck - 1) & 1, abort_flag, p.err)))) {
      fence_after_sync();
      // the segment's start gradient dS0 ([d_v][d_k])
      float* sg = p.sgrad + ((size_t)seg * p.H + h) * kD * kD;
#pragma unroll 1
      for (int cc = 0; cc < kWkCw / 32; ++cc) {
        tmem_ld32(tmem + lrow + col0 + cc * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 32; ++q) sg[(col0 + cc * 32 + q) * kD + r] = __uint_as_float(v[q]);
      }
    }
  }

  __syncwarp();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == kWkEpiWarps + 1) tmem_dealloc(tmem, 256);
}

// ---------------------------------------------------------------------------
// Chunk-local gradients of one (chunk, head) on the tensor core.  With the
// chunk's tokens t, s < L <= 64, gam = the in-chunk cumulative log decay,
// Gam_ts = e^{gam_t - gam_s}, ek_t = e^{gam_{L-1} - gam_t}, B_U = diag(beta) V,
// B_W = diag(beta e^gam) K, A_ts = beta_t Gam_ts k_t . k_s (s < t), T =
// (I + A)^{-1}, and the walk's dS_n and dV' (dU^ = dV'):
//   dQ~ = dO S0^T                   dW = -dV' S0^T        V' = U^ - W S0
//   dK~ = V' dS_n^T                 dP = dO V'^T (s <= t)
//   dT  = dV' B_U^T + dW B_W^T      dA = -lower(T^T dT T^T)
//   dq  = scale e^gam dQ~ + scale (dP o Gam) K
//   dk  = ek dK~ + scale (dP o Gam)^T Q + (M + M^T) K + beta e^gam T^T dW,
//         M_ts = dA_ts beta_t Gam_ts
//   dv  = beta T^T dV'
// and the beta / gam terms of each factor (row and column sums of elementwise
// products).  Each of dq, dk, dv is one TMEM accumulator: its first product
// lands there and the others are added by MMAs whose A rows carry the row
// factors (dq_t = scale e^{gam_t} (dQ~_t + sum_s e^{-gam_s} dP_ts k_s), dk_t =
// ek_t (dK~_t + ...)), so nothing is re-read from memory.  Products with 64
// rows run as M = 128 MMAs whose rows 64-127 read padding and are not used.
// T comes from forward substitution on the CUDA cores.  One CTA of 128
// threads (thread = TMEM lane), thread 0 issues the MMAs; the stages below
// are separated by MMA commits and block barriers.
constexpr int kCkThreads = 128;

__device__ __forceinline__ void unpack8(const uint4 r, float* f) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// Dot product of 32 float32 values with columns 32 cc .. 32 cc + 31 of row
// `row` of a 128-byte-swizzled bf16 tile with `rows` rows.
__device__ __forceinline__ float dot32_sw(const uint8_t* tile, int rows, int row, int cc, const uint32_t* v) {
  float d = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int c8 = cc * 4 + j;
    const uint4 r = *reinterpret_cast<const uint4*>(tile + (c8 >> 3) * rows * 128 + row * 128 +
                                                    (((c8 & 7) ^ (row & 7)) << 4));
    float f[8];
    unpack8(r, f);
#pragma unroll
    for (int k = 0; k < 8; ++k) d = fmaf(__uint_as_float(v[8 * j + k]), f[k], d);
  }
  return d;
}
// shared memory (1024-aligned): bf16 operand tiles, 128-byte swizzled in
// 64-column halves (half stride = rows x 128 bytes)
constexpr int kCkYQ = 0, kCkYK = 16384, kCkYV = 32768;      // q^, k^, v [64][128]
constexpr int kCkDODV = 49152;                                // [dO ; dV'] [128][128]
constexpr int kCkVP = 81920, kCkDW = 98304;                   // V', dW [64][128]
constexpr int kCkR = 114688;                                  // phase region
constexpr int kCkS0 = kCkR, kCkDS = kCkR + 32768, kCkW = kCkR + 65536;   // S0, dS_n [128][128], W [64][128]
constexpr int kCkTb = kCkR, kCkDT = kCkR + 8192, kCkYb = kCkR + 16384, kCkAq = kCkR + 24576,
              kCkAa = kCkR + 32768, kCkAb = kCkR + 40960, kCkAc = kCkR + 49152;   // [64][64] tiles
// float32 [64][64] scratch, element (r, c) at r * 64 + (c ^ (r % 32)) (conflict-free
// rows and columns); F3 in the phase region, F4 over V' and F5 over v (both
// read by the stage-B MMAs only), F1 (GK) and F2 (T) for the whole kernel
constexpr int kCkF3 = kCkR + 57344, kCkF4 = kCkVP, kCkF5 = kCkYV;
constexpr int kCkF1 = kCkR + 81920, kCkF2 = kCkF1 + 16384;
constexpr int kCkSc = kCkF2 + 16384;                          // scalars: gam eg ek beta dgam dbeta misc [64] each
constexpr int kCkBar = kCkSc + 7 * 64 * 4;
constexpr int kCkSmem = kCkBar + 64;
static_assert(kCkF3 + 16384 <= kCkF1 && kCkSmem <= 232448, "chunk kernel shared memory");
__device__ __forceinline__ int fx(int r, int c) { return r * 64 + (c ^ (r & 31)); }
enum { K_A = 0, K_B = 1, K_C = 2, K_D = 3, K_E = 4, K_COUNT = 5 };

// descriptor low words of operand tiles: K-major with `rows` rows (slice kk of
// 16 columns), MN-major with `rows` rows = K (slice kk of 16 rows)
__device__ __forceinline__ uint32_t kmaj(uint32_t base, int rows, int kk) {
  return desc_lo_kmajor(base + (kk >> 2) * rows * 128 + (kk & 3) * 32);
}
__device__ __forceinline__ uint32_t mnmaj(uint32_t base, int rows, int kk) {
  return ((base + kk * 2048) & 0x3FFFFu) >> 4 | (((uint32_t)(rows * 128) >> 4) << 16);
}

__global__ void __launch_bounds__(kCkThreads, 1) gdn_bwd_chunk_kernel(const GbParams p) {
  extern __shared__ __align__(1024) uint8_t csm[];
  const uint32_t sb = smem_u32(csm);
  float* F1 = reinterpret_cast<float*>(csm + kCkF1);   // GK_ts = Gam_ts k_t . k_s (s < t < L)
  float* F2 = reinterpret_cast<float*>(csm + kCkF2);   // T
  float* F3 = reinterpret_cast<float*>(csm + kCkF3);
  float* F4 = reinterpret_cast<float*>(csm + kCkF4);
  float* F5 = reinterpret_cast<float*>(csm + kCkF5);
  float* gam = reinterpret_cast<float*>(csm + kCkSc);
  float* eg = gam + 64;
  float* ek = eg + 64;
  float* bt = ek + 64;
  float* dgam = bt + 64;
  float* dbt = dgam + 64;
  float* misc = dbt + 64;   // per-warp partials: [0..3] <dS_n, S0>, [4..5] the dK~ term
  uint64_t* bars = reinterpret_cast<uint64_t*>(csm + kCkBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + K_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ch = p.chunk0 + (int)(blockIdx.x / p.H), h = (int)(blockIdx.x % p.H);
  const int x0 = p.chunk_start[ch], L = p.chunk_len[ch];
  const size_t row = (size_t)ch * p.H + h;
  const int Hd = p.H * kD;
  const float sc = p.scale;
  const uint32_t lrow = (uint32_t)(warp * 32) << 16;
  // TMEM columns: dq 0-127, dk 128-255 (first V' = W S0), 256-319 KK then dP
  // then dA', 320-383 R1 = dV' V^T, 384-447 R2 = dW K^T (320-447 later dv),
  // 448-511 Y = T^T dT
  constexpr uint32_t cDQ = 0, cDK = 128, cX = 256, cR1 = 320, cR2 = 384, cDV = 320, cY = 448;

  if (tid == 0) {
    for (int b = 0; b < K_COUNT; ++b) mbar_init(&bars[b], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  // ---- loads: q^ k^ v rows, [dO ; dV'], W (bf16 operand tiles); S0 and dS_n
  // rows (thread = d_k row), with the decay term <dS_n, S0>
  {
    const __nv_bfloat16* y = p.y + (size_t)x0 * p.C + h * kD;
#pragma unroll 4
    for (int e = tid; e < 64 * 16; e += kCkThreads) {
      const int t = e >> 4, c8 = e & 15;
      uint4 rq = make_uint4(0, 0, 0, 0), rk = rq, rv = rq, rw = rq;
      if (t < L) {
        const __nv_bfloat16* yr = y + (size_t)t * p.C + c8 * 8;
        rq = *reinterpret_cast<const uint4*>(yr);
        rk = *reinterpret_cast<const uint4*>(yr + Hd);
        rv = *reinterpret_cast<const uint4*>(yr + 2 * Hd);
      }
      rw = *reinterpret_cast<const uint4*>(p.wq + (row * 128 + kC + t) * kD + c8 * 8);   // zero rows past L
      st_sw8(csm + kCkYQ, 64, t, c8, rq);
      st_sw8(csm + kCkYK, 64, t, c8, rk);
      st_sw8(csm + kCkYV, 64, t, c8, rv);
      st_sw8(csm + kCkW, 64, t, c8, rw);
      float f[8];
      if (t < L) {
        const float4* src = reinterpret_cast<const float4*>(p.d_o + ((size_t)(x0 + t) * p.H + h) * kD + c8 * 8);
        const float4 a = src[0], b = src[1];
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) f[k] = 0.f;
      }
      st_sw8(csm + kCkDODV, 128, t, c8, pack8(f));
    }
    // dV' rows from [d_v][64]: thread = (token, half of the d_v columns)
    {
      const float* dvp = p.dvp + row * kC * kD;
      const int t = tid & 63, c0 = (tid >> 6) * 8;
      float f[64];
#pragma unroll
      for (int k = 0; k < 64; ++k) f[k] = dvp[(c0 * 8 + k) * kC + t];
#pragma unroll
      for (int j = 0; j < 8; ++j) st_sw8(csm + kCkDODV, 128, kC + t, c0 + j, pack8(f + 8 * j));
    }
    // S0 row r and dS_n row r (both stored [d_v][d_k]: thread r reads column r)
    const int r = tid;
    const float* s0t = p.s0 + row * kD * kD;
    const float* dse = p.dsend + row * kD * kD;
    float dot = 0.f;
#pragma unroll 1
    for (int c32 = 0; c32 < 4; ++c32) {
      float fs[32], fd[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        fs[k] = s0t[(c32 * 32 + k) * kD + r];
        fd[k] = dse[(c32 * 32 + k) * kD + r];
      }
#pragma unroll
      for (int k = 0; k < 32; ++k) dot = fmaf(fs[k], fd[k], dot);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        st_sw8(csm + kCkS0, 128, r, c32 * 4 + j, pack8(fs + 8 * j));
        st_sw8(csm + kCkDS, 128, r, c32 * 4 + j, pack8(fd + 8 * j));
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
    if (tid < 64) {
      dgam[tid] = 0.f;
      dbt[tid] = 0.f;
    }
    if (lane == 0) misc[warp] = dot;
  }
  if (tid < 32) {   // gam = inclusive prefix sum of g over the chunk; beta; e^gam; e^{gam_{L-1} - gam}
    float a = tid < L ? p.g[(size_t)(x0 + tid) * p.H + h] : 0.f;
    float b = tid + 32 < L ? p.g[(size_t)(x0 + tid + 32) * p.H + h] : 0.f;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float ua = __shfl_up_sync(0xffffffffu, a, off), ub = __shfl_up_sync(0xffffffffu, b, off);
      if (tid >= off) {
        a += ua;
        b += ub;
      }
    }
    b += __shfl_sync(0xffffffffu, a, 31);
    const float gl = __shfl_sync(0xffffffffu, (L - 1) < 32 ? a : b, (L - 1) & 31);
    gam[tid] = a;
    gam[tid + 32] = b;
    eg[tid] = expf(a);
    eg[tid + 32] = expf(b);
    ek[tid] = expf(gl - a);
    ek[tid + 32] = expf(gl - b);
    bt[tid] = tid < L ? p.beta[(size_t)(x0 + tid) * p.H + h] : 0.f;
    bt[tid + 32] = tid + 32 < L ? p.beta[(size_t)(x0 + tid + 32) * p.H + h] : 0.f;
  }
  fence_proxy_async_smem();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  // ---- stage A: [dQ~ ; -dW] = [dO ; dV'] S0^T, W S0, K K^T
  if (tid == 0) {
    constexpr uint32_t id_kk = idesc_bf16(128, 128, 0, 0), id_kmn = idesc_bf16(128, 128, 0, 1);
    constexpr uint32_t id_kk64 = idesc_bf16(128, 64, 0, 0);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_ss_lo(tmem + cDQ, kmaj(sb + kCkDODV, 128, kk), kmaj(sb + kCkS0, 128, kk), id_kk, kk > 0);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_ss_lo(tmem + cDK, kmaj(sb + kCkW, 64, kk), mnmaj(sb + kCkS0, 128, kk), id_kmn, kk > 0);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_ss_lo(tmem + cX, kmaj(sb + kCkYK, 64, kk), kmaj(sb + kCkYK, 64, kk), id_kk64, kk > 0);
    mma_commit(&bars[K_A]);
  }
  bool ok = __all_sync(0xffffffffu, mbar_wait(&bars[K_A], 0, abort_flag, p.err));
  fence_after_sync();
  uint32_t v[32];
  if (ok) {
    if (tid < 64) {
      const int t = tid;
      // dgam_t += scale e^{gam_t} dQ~_t . q_t (q row t from its operand tile)
      float dq = 0.f;
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        tmem_ld32(tmem + cDQ + lrow + cc * 32, v);
        tmem_ld_wait();
        dq += dot32_sw(csm + kCkYQ, 64, t, cc, v);
      }
      if (t < L) dgam[t] += sc * eg[t] * dq;
      // V' = U^ - W S0 -> operand tile
      const float* ut = p.ut + row * kD * kC;
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        tmem_ld32(tmem + cDK + lrow + cc * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float f[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int col = cc * 32 + 8 * j + k;
            f[k] = ut[col * kC + t] - __uint_as_float(v[8 * j + k]);
          }
          st_sw8(csm + kCkVP, 64, t, cc * 4 + j, pack8(f));
        }
      }
      // GK_ts = Gam_ts (k_t . k_s), s < t < L
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {
        tmem_ld32(tmem + cX + lrow + cc * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          const int s = cc * 32 + q;
          F1[fx(t, s)] = (s < t && t < L) ? __expf(gam[t] - gam[s]) * __uint_as_float(v[q]) : 0.f;
        }
      }
    } else {
      // dW = -(dV' S0^T) -> operand tile (rows 64-127 of the stacked product)
      const int t = tid - 64;
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        tmem_ld32(tmem + cDQ + lrow + cc * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float f[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) f[k] = -__uint_as_float(v[8 * j + k]);
          st_sw8(csm + kCkDW, 64, t, cc * 4 + j, pack8(f));
        }
      }
    }
  }
  fence_proxy_async_smem();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();

  // ---- stage B: dK~ = V' dS_n^T (into dk), dP = dO V'^T, R1 = dV' V^T, R2 = dW K^T;
  // meanwhile T = (I + A)^{-1}, A_ts = beta_t GK_ts, one column per thread
  if (ok && tid == 0) {
    constexpr uint32_t id_kk = idesc_bf16(128, 128, 0, 0), id_kk64 = idesc_bf16(128, 64, 0, 0);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_ss_lo(tmem + cDK, kmaj(sb + kCkVP, 64, kk), kmaj(sb + kCkDS, 128, kk), id_kk, kk > 0);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_ss_lo(tmem + cX, kmaj(sb + kCkDODV, 128, kk), kmaj(sb + kCkVP, 64, kk), id_kk64, kk > 0);
    // dV' = rows 64-127 of [dO ; dV']: start 64 rows into each half
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_ss_lo(tmem + cR1, kmaj(sb + kCkDODV + 64 * 128, 128, kk), kmaj(sb + kCkYV, 64, kk), id_kk64, kk > 0);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_ss_lo(tmem + cR2, kmaj(sb + kCkDW, 64, kk), kmaj(sb + kCkYK, 64, kk), id_kk64, kk > 0);
    mma_commit(&bars[K_B]);
  }
  if (tid < 64) {
    // column j of T in registers: T_tj = [t == j] - beta_t sum_{s < t} GK_ts T_sj
    // (T_sj = 0 for s < j, so every row is summed over s < t)
    const int j = tid;
    float X[64];
#pragma unroll
    for (int t = 0; t < 64; ++t) {
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int s = 0; s < t; s += 2) {
        a0 = fmaf(F1[fx(t, s)], X[s], a0);
        if (s + 1 < t) a1 = fmaf(F1[fx(t, s + 1)], X[s + 1], a1);
      }
      X[t] = (t == j ? 1.f : 0.f) - bt[t] * (a0 + a1);
      F2[fx(t, j)] = X[t];
    }
  }
  ok = __all_sync(0xffffffffu, ok && mbar_wait(&bars[K_B], 0, abort_flag, p.err));
  fence_after_sync();
  __syncthreads();   // T complete; the S0 / dS_n / W tiles are no longer read

  // ---- epilogue B (thread t < 64 = row t): the dK~ and dP terms, dT, and the
  // operand tiles of stage C
  float myc = 0.f;   // ek_t dK~_t . k_t
  if (ok && tid < 64) {
    const int t = tid;
    float c = 0.f;
#pragma unroll 1
    for (int cc = 0; cc < 4; ++cc) {
      tmem_ld32(tmem + cDK + lrow + cc * 32, v);
      tmem_ld_wait();
      c += dot32_sw(csm + kCkYK, 64, t, cc, v);
    }
    myc = t < L ? ek[t] * c : 0.f;
    // dP row t (masked s <= t < L) with P row t: E_ts = dP_ts P_ts; Aq, Aa rows
    const uint4* pr4 = reinterpret_cast<const uint4*>(p.pm + (row * kC + t) * kC);
    float esum = 0.f;
#pragma unroll 1
    for (int cc = 0; cc < 2; ++cc) {
      float pf[32];
#pragma unroll
      for (int j = 0; j < 4; ++j) unpack8(pr4[cc * 4 + j], pf + 8 * j);
      tmem_ld32(tmem + cX + lrow + cc * 32, v);
      tmem_ld_wait();
      float aq[32], aa[32];
#pragma unroll
      for (int q = 0; q < 32; ++q) {
        const int s = cc * 32 + q;
        const float dp = (s <= t && t < L) ? __uint_as_float(v[q]) : 0.f;
        const float e = dp * pf[q];
        F5[fx(t, s)] = e;
        esum += e;
        aq[q] = dp * __expf(-gam[s]);
        aa[q] = sc * dp * __expf(gam[t] - gam[L - 1]);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        st_sw8(csm + kCkAq, 64, t, cc * 4 + j, pack8(aq + 8 * j));
        st_sw8(csm + kCkAa, 64, t, cc * 4 + j, pack8(aa + 8 * j));
      }
    }
    dgam[t] += esum;
    // dT_ts = beta_s R1_ts + beta_s e^{gam_s} R2_ts; the T o R1, T o R2 terms
    float r1[32], r2[32];
#pragma unroll 1
    for (int cc = 0; cc < 2; ++cc) {
      tmem_ld32(tmem + cR1 + lrow + cc * 32, v);
      tmem_ld_wait();
#pragma unroll
      for (int q = 0; q < 32; ++q) r1[q] = __uint_as_float(v[q]);
      tmem_ld32(tmem + cR2 + lrow + cc * 32, v);
      tmem_ld_wait();
#pragma unroll
      for (int q = 0; q < 32; ++q) r2[q] = __uint_as_float(v[q]);
      float dt[32];
#pragma unroll
      for (int q = 0; q < 32; ++q) {
        const int s = cc * 32 + q;
        dt[q] = bt[s] * (r1[q] + eg[s] * r2[q]);
        const float T_ts = F2[fx(t, s)];
        F3[fx(t, s)] = T_ts * r1[q];
        F4[fx(t, s)] = T_ts * r2[q];
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) st_sw8(csm + kCkDT, 64, t, cc * 4 + j, pack8(dt + 8 * j));
    }
    // T (bf16, rows s) and Ac (MN-major: row s holds beta_t e^{2 gam_t - gam_{L-1}} T_st)
    {
      float tb[64], ac[64];
#pragma unroll
      for (int u = 0; u < 64; ++u) {
        tb[u] = F2[fx(t, u)];
        ac[u] = tb[u] * bt[u] * __expf(2.f * gam[u] - gam[L - 1]);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        st_sw8(csm + kCkTb, 64, t, j, pack8(tb + 8 * j));
        st_sw8(csm + kCkAc, 64, t, j, pack8(ac + 8 * j));
      }
    }
  }
  {   // dgam: the dK~ term (sum over rows to L-1, minus its own row)
    float c = myc;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) c += __shfl_xor_sync(0xffffffffu, c, off);
    if (tid < 64) {
      dgam[tid] -= myc;
      if (lane == 0) misc[4 + warp] = c;
    }
  }
  fence_proxy_async_smem();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (tid < 64) {   // column sums: the P term of dgam, and the B_U / B_W terms of dbeta, dgam
    const int u = tid;
    float e = 0.f, a1 = 0.f, a2 = 0.f;
    for (int s = 0; s < 64; ++s) {
      e += F5[fx(s, u)];
      a1 += F3[fx(s, u)];
      a2 += F4[fx(s, u)];
    }
    dgam[u] += -e + bt[u] * eg[u] * a2;
    dbt[u] += a1 + eg[u] * a2;
  }

  // ---- stage C: Y = T^T dT; dq += Aq K; dk += Aa Q + Ac dW
  if (ok && tid == 0) {
    constexpr uint32_t id_mm64 = idesc_bf16(128, 64, 1, 1), id_kmn = idesc_bf16(128, 128, 0, 1),
                       id_mmn = idesc_bf16(128, 128, 1, 1);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_ss_lo(tmem + cY, mnmaj(sb + kCkTb, 64, kk), mnmaj(sb + kCkDT, 64, kk), id_mm64, kk > 0);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_ss_lo(tmem + cDQ, kmaj(sb + kCkAq, 64, kk), mnmaj(sb + kCkYK, 64, kk), id_kmn, 1u);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_ss_lo(tmem + cDK, mnmaj(sb + kCkAa, 64, kk), mnmaj(sb + kCkYQ, 64, kk), id_mmn, 1u);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_ss_lo(tmem + cDK, mnmaj(sb + kCkAc, 64, kk), mnmaj(sb + kCkDW, 64, kk), id_mmn, 1u);
    mma_commit(&bars[K_C]);
  }
  ok = __all_sync(0xffffffffu, ok && mbar_wait(&bars[K_C], 0, abort_flag, p.err));
  fence_after_sync();
  if (ok && tid < 64) {
    const int t = tid;
#pragma unroll 1
    for (int cc = 0; cc < 2; ++cc) {
      tmem_ld32(tmem + cY + lrow + cc * 32, v);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 4; ++j) st_sw8(csm + kCkYb, 64, t, cc * 4 + j, pack8(reinterpret_cast<const float*>(v) + 8 * j));
    }
  }
  fence_proxy_async_smem();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();

  // ---- stage D: dA' = Y T^T;  dA = -dA' on s < t < L
  if (ok && tid == 0) {
    constexpr uint32_t id_kk64 = idesc_bf16(128, 64, 0, 0);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_ss_lo(tmem + cX, kmaj(sb + kCkYb, 64, kk), kmaj(sb + kCkTb, 64, kk), id_kk64, kk > 0);
    mma_commit(&bars[K_D]);
  }
  ok = __all_sync(0xffffffffu, ok && mbar_wait(&bars[K_D], 0, abort_flag, p.err));
  fence_after_sync();
  if (ok && tid < 64) {
    const int t = tid;
    float ga = 0.f, gb = 0.f;
#pragma unroll 1
    for (int cc = 0; cc < 2; ++cc) {
      tmem_ld32(tmem + cX + lrow + cc * 32, v);
      tmem_ld_wait();
#pragma unroll
      for (int q = 0; q < 32; ++q) {
        const int s = cc * 32 + q;
        const float da = (s < t && t < L) ? -__uint_as_float(v[q]) : 0.f;
        const float gk = F1[fx(t, s)];
        ga += da * bt[t] * gk;                    // dA_ts A_ts
        gb += da * gk;                            // dbeta term
        F3[fx(t, s)] = da * bt[t] * __expf(gam[t] - gam[s]);   // M_ts
        F4[fx(t, s)] = da * bt[t] * gk;
      }
    }
    dgam[t] += ga;
    dbt[t] += gb;
  }
  __syncthreads();
  if (ok && tid < 64) {
    const int t = tid;
    float col = 0.f, ab[64];
    const float et = __expf(gam[t] - gam[L - 1]);
#pragma unroll
    for (int s = 0; s < 64; ++s) {
      col += F4[fx(s, t)];
      ab[s] = et * (F3[fx(t, s)] + F3[fx(s, t)]);
    }
    dgam[t] -= col;
#pragma unroll
    for (int j = 0; j < 8; ++j) st_sw8(csm + kCkAb, 64, t, j, pack8(ab + 8 * j));
  }
  fence_proxy_async_smem();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();

  // ---- stage E: dk += Ab K;  dv = T^T dV'
  if (ok && tid == 0) {
    constexpr uint32_t id_kmn = idesc_bf16(128, 128, 0, 1), id_mmn = idesc_bf16(128, 128, 1, 1);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_ss_lo(tmem + cDK, kmaj(sb + kCkAb, 64, kk), mnmaj(sb + kCkYK, 64, kk), id_kmn, 1u);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_ss_lo(tmem + cDV, mnmaj(sb + kCkTb, 64, kk), mnmaj(sb + kCkDODV + 64 * 128, 128, kk), id_mmn, kk > 0);
    mma_commit(&bars[K_E]);
  }
  ok = __all_sync(0xffffffffu, ok && mbar_wait(&bars[K_E], 0, abort_flag, p.err));
  fence_after_sync();
  if (ok && tid < 64) {
    // TMEM loads are warp-collective: every lane loads, rows t < L are stored
    const int t = tid;
    float* dqo = p.dqkv + (size_t)(x0 + t) * p.C + h * kD;
    const float fq = sc * eg[t], fk = ek[t], fv = bt[t];
#pragma unroll 1
    for (int part = 0; part < 3; ++part) {
      const uint32_t col0 = part == 0 ? cDQ : part == 1 ? cDK : cDV;
      const float f = part == 0 ? fq : part == 1 ? fk : fv;
      float4* dst = reinterpret_cast<float4*>(dqo + part * Hd);
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        tmem_ld32(tmem + col0 + lrow + cc * 32, v);
        tmem_ld_wait();
        if (t < L)
#pragma unroll
          for (int q = 0; q < 8; ++q)
            dst[cc * 8 + q] = make_float4(f * __uint_as_float(v[4 * q]), f * __uint_as_float(v[4 * q + 1]),
                                          f * __uint_as_float(v[4 * q + 2]), f * __uint_as_float(v[4 * q + 3]));
      }
    }
  }
  __syncthreads();
  if (tid == 0)   // the terms of row L-1 summed over rows or warps: the dK~ term, then the decay term
    dgam[L - 1] += (misc[4] + misc[5]) + eg[L - 1] * (((misc[0] + misc[1]) + misc[2]) + misc[3]);
  __syncthreads();
  if (ok && tid < 32) {   // dg = reverse cumulative sum of dgam over the chunk's tokens; dbeta
    float a = tid + 32 < L ? dgam[tid + 32] : 0.f, b = tid < L ? dgam[tid] : 0.f;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float ua = __shfl_down_sync(0xffffffffu, a, off), ub = __shfl_down_sync(0xffffffffu, b, off);
      if (tid + off < 32) {
        a += ua;
        b += ub;
      }
    }
    b += __shfl_sync(0xffffffffu, a, 0);
    if (tid < L) {
      p.dg[(size_t)(x0 + tid) * p.H + h] = b;
      p.dbeta[(size_t)(x0 + tid) * p.H + h] = dbt[tid];
    }
    if (tid + 32 < L) {
      p.dg[(size_t)(x0 + tid + 32) * p.H + h] = a;
      p.dbeta[(size_t)(x0 + tid + 32) * p.H + h] = dbt[tid + 32];
    }
  }
  if (!ok && tid == 0) atomicOr(p.err, kErrTimeout);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------------------
// Back through the unit-norm heads and SiLU: dz of every (token, channel),
// written over dy; and the block's share of the weight gradient,
// dw[c][tap] = sum over its tokens of x[source of the tap] dz.  Unit = (64
// tokens, one group of 128 channels: a q, k or v head); thread = (4 tokens,
// 8 channels), so the 16 lanes of one token hold one head.
// A CTA keeps one channel group (its weights in registers) and walks token
// blocks bx0, bx0 + S, ...: per block one TMA copy brings the x rows
// xb-3 .. xb+63 of the group (bf16, zero rows outside the tensor) and one the
// block's dy^ rows (f32), the next block's copies in flight while this one
// is computed.  Per block the weight-gradient share is summed in a fixed
// order (the two token lanes of a warp, then the warps) and written to the
// block's slot, so the sum over blocks stays in block order.
constexpr int kTkRows = 64 + 3;
constexpr int kTkX = kTkRows * kD * 2;      // x rows, bf16
constexpr int kTkY = 64 * kD * 4;           // dy^ rows, f32
constexpr int kTkBuf = kTkX + kTkY;
constexpr int kTkRed = (kBT / 32) * 16 * 33 * 4;   // [warp][vector][8 channels x 4 taps (+1)]
constexpr int kTkSmem = 2 * kTkBuf + kTkRed + 64;

__global__ void __launch_bounds__(kBT, 1) gdn_bwd_token_kernel(const __grid_constant__ CUtensorMap mx,
                                                               const __grid_constant__ CUtensorMap my,
                                                               const GbParams p, int S) {
  extern __shared__ __align__(128) uint8_t tsm[];
  float* red = reinterpret_cast<float*>(tsm + 2 * kTkBuf);
  uint64_t* bars = reinterpret_cast<uint64_t*>(tsm + 2 * kTkBuf + kTkRed);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2);
  __shared__ int taps[2][64][3];
  const int G = 3 * p.H, nbx = (p.N + 63) / 64;
  const int grp = blockIdx.x % G, bx0 = blockIdx.x / G;
  const int warp = threadIdx.x >> 5, lt = threadIdx.x >> 4, vec = threadIdx.x & 15;
  const int ch = grp * kD + vec * 8;
  const bool is_qk = grp < 2 * p.H;
  const unsigned grpmask = 0xffffu << (threadIdx.x & 16);
  auto issue = [&](int bx, int buf) {
    mbar_expect_tx(&bars[buf], kTkBuf);
    tma_load_2d(tsm + buf * kTkBuf, &mx, &bars[buf], grp * kD, bx * 64 - 3);
    tma_load_2d(tsm + buf * kTkBuf + kTkX, &my, &bars[buf], grp * kD, bx * 64);
  };
  auto load_taps = [&](int bx, int& t0, int& t1, int& t2) {
    const int x = bx * 64 + threadIdx.x;
    const bool in = x < p.N;
    t0 = in ? p.prev[x] : -2;
    t1 = in ? p.prev2[x] : -1;
    t2 = in ? p.prev3[x] : -1;
  };
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    *abort_flag = 0;
    fence_mbar_init();
    if (bx0 < nbx) issue(bx0, 0);
  }
  if (threadIdx.x < 64 && bx0 < nbx) load_taps(bx0, taps[0][threadIdx.x][0], taps[0][threadIdx.x][1], taps[0][threadIdx.x][2]);
  float4 wv[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) wv[i] = reinterpret_cast<const float4*>(p.conv_w)[ch + i];
  __syncthreads();
  int j = 0;
  for (int bx = bx0; bx < nbx; bx += S, ++j) {
    const int buf = j & 1, nb = bx + S;
    int n0 = -2, n1 = -1, n2 = -1;
    if (nb < nbx) {   // the next block (that buffer was freed by the barrier ending the previous block)
      if (threadIdx.x == 0) issue(nb, buf ^ 1);
      if (threadIdx.x < 64) load_taps(nb, n0, n1, n2);
    }
    if (!__syncthreads_and(mbar_wait(&bars[buf], (j >> 1) & 1, abort_flag, p.err))) {
      mbar_wait_drain(&bars[buf], (j >> 1) & 1);
      if (nb < nbx) mbar_wait_drain(&bars[buf ^ 1], ((j + 1) >> 1) & 1);
      return;
    }
    const int xb = bx * 64;
    const uint8_t* xt = tsm + buf * kTkBuf;
    const float* yt = reinterpret_cast<const float*>(tsm + buf * kTkBuf + kTkX);
    float dw[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int t = 0; t < 4; ++t) dw[i][t] = 0.f;
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      const int tl = it * 16 + lt, x = xb + tl;
      const int p1 = taps[buf][tl][0];
      const bool real = p1 != -2;   // the same for all 16 lanes of the token
      const int src[4] = {taps[buf][tl][2], taps[buf][tl][1], p1, x};
      float xin[4][8], z[8];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        uint4 r = make_uint4(0, 0, 0, 0);
        if (real && src[t] >= 0) {
          const int rr = src[t] - (xb - 3);
          r = (rr >= 0 && rr < kTkRows) ? *reinterpret_cast<const uint4*>(xt + rr * (kD * 2) + vec * 16)
                                        : *reinterpret_cast<const uint4*>(p.x + (size_t)src[t] * p.C + ch);
        }
        unpack8(r, xin[t]);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i)
        z[i] = fmaf(wv[i].x, xin[0][i], fmaf(wv[i].y, xin[1][i], fmaf(wv[i].z, xin[2][i], wv[i].w * xin[3][i])));
      float dy[8];
      {
        const float4 da = *reinterpret_cast<const float4*>(yt + tl * kD + vec * 8);
        const float4 db = *reinterpret_cast<const float4*>(yt + tl * kD + vec * 8 + 4);
        const float d8[8] = {da.x, da.y, da.z, da.w, db.x, db.y, db.z, db.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) dy[i] = real ? d8[i] : 0.f;
      }
      float sg[8], y[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        sg[i] = __fdividef(1.f, 1.f + __expf(-z[i]));
        y[i] = z[i] * sg[i];
      }
      if (is_qk) {   // y^ = y / n,  dy = (dy^ - y^ (y^ . dy^)) / n
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) ss = fmaf(y[i], y[i], ss);
        ss += __shfl_xor_sync(grpmask, ss, 8);
        ss += __shfl_xor_sync(grpmask, ss, 4);
        ss += __shfl_xor_sync(grpmask, ss, 2);
        ss += __shfl_xor_sync(grpmask, ss, 1);
        const float rn = rsqrtf(ss + 1e-6f);
        float dot = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) dot = fmaf(y[i] * rn, dy[i], dot);
        dot += __shfl_xor_sync(grpmask, dot, 8);
        dot += __shfl_xor_sync(grpmask, dot, 4);
        dot += __shfl_xor_sync(grpmask, dot, 2);
        dot += __shfl_xor_sync(grpmask, dot, 1);
#pragma unroll
        for (int i = 0; i < 8; ++i) dy[i] = (dy[i] - y[i] * rn * dot) * rn;
      }
      if (!real) continue;
      float dz[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        dz[i] = dy[i] * sg[i] * (1.f + z[i] * (1.f - sg[i]));
#pragma unroll
        for (int t = 0; t < 4; ++t) dw[i][t] = fmaf(xin[t][i], dz[i], dw[i][t]);
      }
      float4* o = reinterpret_cast<float4*>(p.dqkv + (size_t)x * p.C + ch);
      o[0] = make_float4(dz[0], dz[1], dz[2], dz[3]);
      o[1] = make_float4(dz[4], dz[5], dz[6], dz[7]);
    }
    // this block's weight-gradient share: the warp's two token lanes (lane
    // and lane ^ 16), then the eight warps in order
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float v = dw[i][t] + __shfl_xor_sync(0xffffffffu, dw[i][t], 16);
        if ((threadIdx.x & 16) == 0) red[(warp * 16 + vec) * 33 + i * 4 + t] = v;
      }
    if (threadIdx.x < 64 && nb < nbx) {
      taps[buf ^ 1][threadIdx.x][0] = n0;
      taps[buf ^ 1][threadIdx.x][1] = n1;
      taps[buf ^ 1][threadIdx.x][2] = n2;
    }
    __syncthreads();
    float* share = p.dwp + ((size_t)bx * p.C + grp * kD) * 4;
    for (int e = threadIdx.x; e < 16 * 32; e += kBT) {
      const int vv = e / 32, q = e % 32;
      float acc = 0.f;
      for (int w = 0; w < kBT / 32; ++w) acc += red[(w * 16 + vv) * 33 + q];
      share[(vv * 8 + q / 4) * 4 + (q % 4)] = acc;
    }
    __syncthreads();   // red and this block's buffers are free for the next block
  }
}


// dx[j] = w3 dz[j] + sum over successors i of (w2 dz[i] + sum over successors
// k of i of (w1 dz[k] + sum over successors l of k of w0 dz[l])): every token
// that reads x[j] through a tap, summed in successor-list order.  A block per
// (64 tokens, channel group of 128); thread = (4 consecutive tokens, 8
// channels); pads get 0.
__global__ void __launch_bounds__(kBT) gdn_bwd_dx_kernel(const GbParams p) {
  // Successor offsets and path predecessors of the block's tokens and the
  // three after them, loaded together: a token whose only successor is the
  // next token (one successor, and the next token's predecessor is it)
  // passes its gradient straight along; inside a segment a token's readers
  // are just the next three tokens, read directly; elsewhere (segment ends,
  // branch points) the successor lists are walked.
  __shared__ int s_off[68], s_prev[68];
  const int grp = blockIdx.y, lt = threadIdx.x >> 4, vec = threadIdx.x & 15;
  const int ch = grp * kD + vec * 8;
  const int x0 = blockIdx.x * 64;
  if (threadIdx.x < 68) {
    const int t = x0 + (int)threadIdx.x;
    s_off[threadIdx.x] = t <= p.N ? p.succ_off[t] : -1;
    s_prev[threadIdx.x] = t < p.N ? p.prev[t] : -2;
  }
  float4 wv[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) wv[i] = reinterpret_cast<const float4*>(p.conv_w)[ch + i];
  __syncthreads();
  auto add = [&](float* acc, int src, int tap) {
    const float* d = p.dqkv + (size_t)src * p.C + ch;
    const float4 a = reinterpret_cast<const float4*>(d)[0], b = reinterpret_cast<const float4*>(d)[1];
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float w = tap == 0 ? wv[i].x : tap == 1 ? wv[i].y : tap == 2 ? wv[i].z : wv[i].w;
      acc[i] = fmaf(w, v[i], acc[i]);
    }
  };
  // thread = (4 consecutive tokens tb .. tb + 3 of the block, 8 channels)
  const int tb = 4 * lt;
  // the only successor of block token i is token i + 1
  auto next_only = [&](int i) { return s_off[i + 1] - s_off[i] == 1 && s_prev[i + 1] == x0 + i; };
  bool plain4 = x0 + tb + 3 < p.N;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int tl = tb + k;
    plain4 = plain4 && s_prev[tl] != -2 && next_only(tl) && next_only(tl + 1) && next_only(tl + 2);
  }
  if (plain4) {
    // Four tokens inside a segment: token k reads rows x + k .. x + k + 3 with
    // taps 3, 2, 1, 0; the 7 rows are taken once, in order, so every token's
    // sum has the order of the general path below.
    const int x = x0 + tb;
    float acc[4][8];
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[k][i] = 0.f;
#pragma unroll
    for (int j = 0; j < 7; ++j) {
      const float4* d = reinterpret_cast<const float4*>(p.dqkv + (size_t)(x + j) * p.C + ch);
      const float4 ra = d[0], rb = d[1];
      const float v[8] = {ra.x, ra.y, ra.z, ra.w, rb.x, rb.y, rb.z, rb.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int q = j - k;   // this row is the token's q-th reader: tap 3 - q
        if (q < 0 || q > 3) continue;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float w = q == 0 ? wv[i].w : q == 1 ? wv[i].z : q == 2 ? wv[i].y : wv[i].x;
          acc[k][i] = fmaf(w, v[i], acc[k][i]);
        }
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float4* out = reinterpret_cast<float4*>(p.dx + (size_t)(x + k) * p.C + ch);
      out[0] = make_float4(acc[k][0], acc[k][1], acc[k][2], acc[k][3]);
      out[1] = make_float4(acc[k][4], acc[k][5], acc[k][6], acc[k][7]);
    }
    return;
  }
#pragma unroll 1
  for (int k = 0; k < 4; ++k) {
    const int tl = tb + k, x = x0 + tl;
    if (x >= p.N) continue;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    if (p.prev[x] != -2) {
      add(acc, x, 3);
      for (int a = p.succ_off[x]; a < p.succ_off[x + 1]; ++a) {
        const int i1 = p.succ[a];
        add(acc, i1, 2);
        for (int b = p.succ_off[i1]; b < p.succ_off[i1 + 1]; ++b) {
          const int i2 = p.succ[b];
          add(acc, i2, 1);
          for (int c = p.succ_off[i2]; c < p.succ_off[i2 + 1]; ++c) add(acc, p.succ[c], 0);
        }
      }
    }
    float4* out = reinterpret_cast<float4*>(p.dx + (size_t)x * p.C + ch);
    out[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    out[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

// dconv_w[c][tap] = the blocks' shares summed in block order; one thread per (c, tap).
__global__ void __launch_bounds__(kBT) gdn_bwd_dw_kernel(const GbParams p, int n_blocks) {
  const int e = blockIdx.x * kBT + threadIdx.x;
  if (e >= p.C * 4) return;
  float a = 0.f;
  for (int b = 0; b < n_blocks; ++b) a += p.dwp[(size_t)b * p.C * 4 + e];
  p.dconv_w[e] = a;
}

// A high-priority stream for the reverse walks and a second one for the chunk
// pass of the deeper chunks, with their events; one set per device.
struct GbStreams {
  bool ready = false;
  cudaStream_t hi = nullptr, aux = nullptr;
  cudaEvent_t fork = nullptr, deep = nullptr, join_hi = nullptr, join_aux = nullptr;
};
std::mutex g_gb_mu;
GbStreams g_gb_streams[64];

cudaError_t gb_streams(GbStreams** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_gb_mu);
  GbStreams& g = g_gb_streams[dev];
  if (!g.ready) {
    int least = 0, greatest = 0;
    e = cudaDeviceGetStreamPriorityRange(&least, &greatest);
    if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&g.hi, cudaStreamNonBlocking, greatest);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&g.aux, cudaStreamNonBlocking);
    for (cudaEvent_t* ev : {&g.fork, &g.deep, &g.join_hi, &g.join_aux})
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    if (e != cudaSuccess) return e;
    g.ready = true;
  }
  *out = &g;
  return cudaSuccess;
}

}  // namespace
}  // namespace stp

using namespace stp;

extern "C" stp_status stp_gdn_bwd(const stp_gdn_desc* desc, const void* plan, const void* d_plan, const void* x,
                                  const float* conv_w, const float* g, const float* beta, const float* d_o,
                                  float* dx, float* dconv_w, float* dg, float* dbeta, void* d_ws, void* stream) {
  clear_error();
  stp_status st = check_gdn_desc(desc);
  if (st) return st;
  const int32_t* w = static_cast<const int32_t*>(plan);
  if ((st = check_gdn_plan(desc, w))) return st;
  if (!d_plan || !x || !conv_w || !g || !beta || !d_o || !dx || !dconv_w || !dg || !dbeta || !d_ws)
    return fail(STP_EINVAL, "stp_gdn_bwd: NULL device pointer");
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(conv_w) | reinterpret_cast<uintptr_t>(d_o) |
       reinterpret_cast<uintptr_t>(dx)) & 15 ||
      (reinterpret_cast<uintptr_t>(d_ws) | reinterpret_cast<uintptr_t>(d_plan)) & 255)
    return fail(STP_EINVAL, "stp_gdn_bwd: x, conv_w, d_o, dx 16-byte, d_plan and ws 256-byte aligned");
  const int N = w[GP_N], H = desc->n_heads, n_chunk = w[GP_NCHUNK], n_seg = w[GP_NSEG], n_depth = w[GP_NDEPTH];
  const int C = 3 * H * kD;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(dconv_w, 0, (size_t)C * 4 * 4, s);
  if (e == cudaSuccess && N > 0) e = cudaMemsetAsync(dg, 0, (size_t)N * H * 4, s);
  if (e == cudaSuccess && N > 0) e = cudaMemsetAsync(dbeta, 0, (size_t)N * H * 4, s);
  if (e != cudaSuccess) return fail(STP_ECUDA, "stp_gdn_bwd: %s", cudaGetErrorString(e));
  if (N == 0) return STP_OK;
  const int32_t* dp = static_cast<const int32_t*>(d_plan);
  char* ws = static_cast<char*>(d_ws);
  const GdnLayout Lw = gdn_layout(N, H, n_chunk, n_seg);
  GbParams p;
  p.N = N;
  p.H = H;
  p.C = C;
  p.seg0 = 0;
  p.chunk0 = 0;
  p.scale = desc->scale;
  p.prev = dp + w[GP_PREV];
  p.prev2 = dp + w[GP_PREV2];
  p.prev3 = dp + w[GP_PREV3];
  p.seg_len = dp + w[GP_SEG_LEN];
  p.seg_chunk0 = dp + w[GP_SEG_CHUNK0];
  p.child_off = dp + w[GP_CHILD_OFF];
  p.child = dp + w[GP_CHILD];
  p.chunk_start = dp + w[GP_CHUNK_START];
  p.chunk_len = dp + w[GP_CHUNK_LEN];
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.conv_w = conv_w;
  p.g = g;
  p.beta = beta;
  p.d_o = d_o;
  p.y = reinterpret_cast<const __nv_bfloat16*>(ws + Lw.y);
  p.wq = reinterpret_cast<const __nv_bfloat16*>(ws + Lw.wq);
  p.kt = reinterpret_cast<const __nv_bfloat16*>(ws + Lw.kt);
  p.pm = reinterpret_cast<const __nv_bfloat16*>(ws + Lw.pm);
  p.ut = reinterpret_cast<const float*>(ws + Lw.ut);
  p.decay = reinterpret_cast<const float*>(ws + Lw.decay);
  p.s0 = reinterpret_cast<const float*>(ws + Lw.s0);
  p.dsend = reinterpret_cast<float*>(ws + Lw.dsend);
  p.dvp = reinterpret_cast<float*>(ws + Lw.dvp);
  p.sgrad = reinterpret_cast<float*>(ws + Lw.sgrad);
  p.dqkv = reinterpret_cast<float*>(ws + Lw.dqkv);
  p.dwp = reinterpret_cast<float*>(ws + Lw.dwp);
  p.succ_off = dp + w[GP_SUCC_OFF];
  p.succ = dp + w[GP_SUCC];
  p.dx = dx;
  p.dconv_w = dconv_w;
  p.dg = dg;
  p.dbeta = dbeta;
  p.err = reinterpret_cast<uint32_t*>(ws);
  CUtensorMap mwq, mkt, mpm, mtx, mty;
  if (!map_rows(&mtx, p.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, N, C, kTkRows) ||
      !map_rows(&mty, p.dqkv, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, N, C, 64))
    return fail(STP_ECUDA, "stp_gdn_bwd: tensor map encoding failed");
  if (n_chunk > 0 &&
      (!map_2d(&mwq, p.wq, (int64_t)n_chunk * H * 128, kD, 128) ||
       !map_2d(&mkt, p.kt, (int64_t)n_chunk * H * kC, kD, kC) ||
       !map_2d(&mpm, p.pm, (int64_t)n_chunk * H * kC, kC, kC)))
    return fail(STP_ECUDA, "stp_gdn_bwd: tensor map encoding failed");
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(gdn_bwd_walk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kWkSmem);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(gdn_bwd_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kCkSmem);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(gdn_bwd_token_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTkSmem);
  });
  if (attr_err != cudaSuccess) return fail(STP_ECUDA, "stp_gdn_bwd: %s", cudaGetErrorString(attr_err));
  // pads keep dq^, dk^, dv = 0 (the chunk kernel writes real tokens only)
  e = cudaMemsetAsync(p.dqkv, 0, (size_t)N * C * 4, s);
  if (e != cudaSuccess) return fail(STP_ECUDA, "stp_gdn_bwd: %s", cudaGetErrorString(e));
  const int32_t* depth_off = w + w[GP_DEPTH_OFF];
  const int32_t* seg_chunk0 = w + w[GP_SEG_CHUNK0];
  auto walk = [&](int d, cudaStream_t st) {
    const int n = depth_off[d + 1] - depth_off[d];
    if (n <= 0) return;
    GbParams q = p;
    q.seg0 = depth_off[d];
    gdn_bwd_walk_kernel<<<(unsigned)(n * H), kWkThreads, kWkSmem, st>>>(mwq, mkt, mpm, q);
  };
  auto chunks = [&](int c_begin, int c_end, cudaStream_t st) {   // the chunk pass over chunks [c_begin, c_end)
    if (c_end <= c_begin) return;
    GbParams q = p;
    q.chunk0 = c_begin;
    gdn_bwd_chunk_kernel<<<(unsigned)((c_end - c_begin) * H), kCkThreads, kCkSmem, st>>>(q);
  };
  // Chunks are numbered depth by depth.  With three depths or more, the chunk
  // pass over the chunks of depth 2 and below starts on a second stream once
  // their walks are done, beside the walks of depths 1 and 0 (one CTA per
  // head and segment: a few SMs), which run on a high-priority stream.
  const int c2 = n_depth > 2 ? seg_chunk0[depth_off[2]] : n_chunk;   // first chunk below depth 1
  if (c2 < n_chunk) {
    GbStreams* gs = nullptr;
    if ((e = gb_streams(&gs)) != cudaSuccess) return fail(STP_ECUDA, "stp_gdn_bwd: %s", cudaGetErrorString(e));
    std::lock_guard<std::mutex> lock(g_gb_mu);
    e = cudaEventRecord(gs->fork, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(gs->hi, gs->fork, 0);
    if (e == cudaSuccess) {
      for (int d = n_depth - 1; d >= 2; --d) walk(d, gs->hi);
      e = cudaEventRecord(gs->deep, gs->hi);
    }
    if (e == cudaSuccess) e = cudaStreamWaitEvent(gs->aux, gs->deep, 0);
    if (e == cudaSuccess) {
      chunks(c2, n_chunk, gs->aux);
      e = cudaEventRecord(gs->join_aux, gs->aux);
    }
    if (e == cudaSuccess) {
      walk(1, gs->hi);
      walk(0, gs->hi);
      chunks(0, c2, gs->hi);
      e = cudaEventRecord(gs->join_hi, gs->hi);
    }
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, gs->join_hi, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, gs->join_aux, 0);
    if (e != cudaSuccess) return fail(STP_ECUDA, "stp_gdn_bwd: %s", cudaGetErrorString(e));
  } else {
    for (int d = n_depth - 1; d >= 0; --d) walk(d, s);
    chunks(0, n_chunk, s);
  }
  const unsigned n_blocks = (unsigned)((N + 63) / 64);
  {
    // a CTA per (channel group, one of S token-block strides)
    static int n_sm = 0;
    if (n_sm == 0) {
      int dev = 0;
      if (cudaGetDevice(&dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n_sm <= 0)
        n_sm = 148;
    }
    const int G = 3 * H;
    const int S = std::max(1, std::min((int)n_blocks, n_sm / G > 0 ? n_sm / G : 1));
    gdn_bwd_token_kernel<<<(unsigned)(G * S), kBT, kTkSmem, s>>>(mtx, mty, p, S);
  }
  gdn_bwd_dx_kernel<<<dim3(n_blocks, (unsigned)(3 * H)), kBT, 0, s>>>(p);
  gdn_bwd_dw_kernel<<<(unsigned)((C * 4 + kBT - 1) / kBT), kBT, 0, s>>>(p, (int)n_blocks);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(STP_ECUDA, "stp_gdn_bwd: %s", cudaGetErrorString(e));
  return STP_OK;
}
