// Tree-aware Gated DeltaNet layer core, forward ("Prefix tree packing", GDN
// section: one pass per tree depth, every segment of that depth at once, a
// child starting from its parent's final state; "ART-Optimized Megatron", the
// GDN paragraphs: the convolution of a branch reads the parent's last inputs).
//
// Per head, with chunk-local cumulative log decay gam_t (t < L <= 64), the
// gated delta rule over a chunk that starts from state S0 ([d_k, d_v]) is
//   A     = strictly lower (beta_t e^{gam_t - gam_s} k_t . k_s)
//   U^    = (I + A)^{-1} diag(beta) V,   W = (I + A)^{-1} diag(beta e^{gam}) K
//   V'    = U^ - W S0
//   O     = scale (diag(e^{gam}) Q S0 + (Q K^T o Gamma) V'),  Gamma_ts = e^{gam_t - gam_s}, s <= t
//   S_L   = e^{gam_L} S0 + (diag(e^{gam_L - gam}) K)^T V'
// (the WY form of the delta rule: substituting the recurrence into itself
// chunk by chunk).  Three kernels (the training forward also writes each
// chunk's starting state S0 for the backward in gdn_bwd.cu):
//   gdn_conv_kernel   persistent, a CTA per (q / k / v head, token-block
//                     stride), 128-token blocks: width-4 causal convolution
//                     along each token's path (prev pointers of the plan; a
//                     block's rows arrive by one TMA copy), SiLU, unit q and k
//                     heads; pads get o = 0.
//   gdn_prep_kernel   one block per (chunk, head): [Q K^T; K K^T] on the tensor
//                     core; T = (I + A)^{-1} of the unit-lower-triangular
//                     system in float32 (two 32 x 32 diagonal blocks by
//                     substitution, the off-diagonal one by two products); then
//                     U^ = T diag(beta) V and W = T diag(beta e^gam) K on the
//                     tensor core (T split into bf16 hi + lo, so the products
//                     keep ~16 bits), and the chunk's operands
//                     [Q~; W] (Q~ = scale e^{gam} Q), K~ = e^{gam_L - gam} K,
//                     P = scale (Q K^T o Gamma) in bf16, U^ transposed in
//                     float32 and e^{gam_L}.  Nothing here depends on a state.
//   gdn_state_kernel  one launch per depth, one CTA per (segment, head): the
//                     state lives in TMEM (float32) for the whole segment; per
//                     chunk the tensor core forms [Q~; W] S0, the epilogue warps
//                     make V' = U^ - W S0, then O += P V' and S += K~^T V' (the
//                     state pre-scaled by e^{gam_L}); the segment's final state
//                     goes to HBM for its children.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "gdn_common.h"
#include "internal.h"
#include "layout.h"
#include "tc_ptx.cuh"

namespace stp {
namespace {

using namespace tc;

constexpr int kGd = 128;          // head dim
constexpr int kGc = kGdnChunk;    // tokens per chunk
constexpr int kConvThreads = 256;
constexpr int kConvPerSm = 2;   // resident convolution CTAs per SM (~100 registers a thread)
constexpr int kPrepThreads = 256;
constexpr int kStThreads = 320;   // warps 0-7 epilogue (a TMEM lane, half its columns), 8 loads, 9 MMA

// gdn_prep_kernel shared memory, from a 1024-byte aligned base: [Q; K] as a
// 128 x 128 bf16 K-major operand (128-byte swizzle, two 64-column halves);
// V bf16 as a 64 x 128 MN-major operand (two 64-column halves of 64 rows);
// A float32 column-major [64][68] (columns 16-byte aligned); the two split
// halves (hi, lo) of [T diag(beta); T diag(beta e^gam)] as 128 x 64 bf16
// K-major operands; gam, beta, e^gam, e^{gam_L - gam} [64]; the MMA barrier
// and the TMEM address.
constexpr int kPrepLa = 68;
constexpr int kPoV = 32768, kPoA = kPoV + 16384, kPoT = 67584, kPoGam = kPoT + 32768, kPoBeta = kPoGam + 256,
              kPoEg = kPoBeta + 256, kPoEk = kPoEg + 256, kPoBar = kPoEk + 256;
constexpr int kPrepSmem = kPoBar + 64 + 1024;
static_assert(kPoA + kGc * kPrepLa * 4 <= kPoT && kPoT % 1024 == 0, "prep shared-memory layout");

// gdn_state_kernel shared memory, from a 1024-byte aligned base.  A stage holds
// [Q~; W] (32 KB), K~ (16 KB) and P (8 KB); P is the top half of a 128-row MMA
// operand whose bottom half is whatever the next 8 KB hold -- it only adds
// to accumulator rows 64-127 (W S0) after they have been read.
constexpr int kStStage = 57344;
constexpr int kOffKt = 32768, kOffP = 49152;
constexpr int kOffSop = 2 * kStStage;           // S0 as a bf16 operand, 32 KB
constexpr int kOffVop = kOffSop + 32768;        // V' as a bf16 operand, 16 KB
constexpr int kOffUt = kOffVop + 16384;         // U^ transposed, float32, 32 KB
constexpr int kOstLd = 528;                     // output staging: 64 rows of 512 B, padded
constexpr int kOffOst = kOffUt + 32768;
constexpr int kOffBar = kOffOst + 64 * kOstLd;
constexpr int kStSmem = kOffBar + 256 + 1024;

struct GdnParams {
  int N, T, H, C, seg0, chunk0;   // T: row length; seg0, chunk0: first segment / chunk of a launch
  float scale;
  const int32_t* prev;      // token 1, 2 and 3 back on the path (-2 on prev: a pad)
  const int32_t* prev2;
  const int32_t* prev3;
  const int32_t* seg_len;
  const int32_t* seg_parent;
  const int32_t* seg_chunk0;
  const int32_t* chunk_start;
  const int32_t* chunk_len;
  const __nv_bfloat16* x;   // [N, C]
  const float* conv_w;      // [C, 4]
  const float* g;           // [N, H]
  const float* beta;        // [N, H]
  __nv_bfloat16* y;         // [N, C]
  __nv_bfloat16* wq;        // [n_chunk H 128, 128]  rows 0-63 Q~, 64-127 W
  __nv_bfloat16* kt;        // [n_chunk H 64, 128]
  __nv_bfloat16* pm;        // [n_chunk H 64, 64]
  float* ut;                // [n_chunk H, 128, 64]
  float* decay;             // [n_chunk H]
  float* state;             // [n_seg H, 128, 128]
  float* s0;                // [n_chunk H, 128 d_v, 128 d_k] each chunk's starting state, or null (inference)
  float* o;                 // [N, H, 128]
  uint32_t* err;
};

enum { B_F = 0, B_E = 2, B_SR = 4, B_M1 = 5, B_VR = 6, B_M2 = 7, B_UF = 8, B_UE = 9, B_DRAIN = 10, B_COUNT = 11 };

typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                             const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                             CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_gdn() {
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

// [rows, cols] bf16 as a 2-D tensor; boxes of 64 columns x box_rows rows, 128-byte swizzled.
bool make_map_2d(CUtensorMap* m, const void* base, int64_t rows, int cols, int box_rows) {
  EncodeFn enc = encode_gdn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// x [rows, cols] bf16 as a 2-D tensor; boxes of 128 columns x kConvRows rows,
// no swizzle (rows of 256 bytes in shared memory).
bool make_map_x(CUtensorMap* m, const void* base, int64_t rows, int cols, int box_rows) {
  EncodeFn enc = encode_gdn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

__device__ __forceinline__ void tma_load_2d_g(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1) {
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

// The same with the halves 16 KB apart (the K rows of the [Q; K] tile).
__device__ __forceinline__ uint32_t desc_lo_mn16k(uint32_t addr) {
  return ((addr & 0x3FFFFu) >> 4) | ((16384u >> 4) << 16);
}

__device__ __forceinline__ void unpack8(const uint4 r, float* f) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// ---------------------------------------------------------------------------
// Path convolution + SiLU + unit q, k heads.  Unit of work = (kConvTok
// tokens, one group of 128 channels: a q, k or v head); thread = (4
// consecutive tokens of each 64, 8 channels), so the 16 lanes of a token hold
// one head.  A CTA keeps one channel group (its weights stay in registers)
// and walks token blocks bx0, bx0 + S, ...; one TMA copy per block brings the
// x rows xb-3 .. xb+kConvTok-1 of the group (zero rows outside the tensor)
// into shared memory, the next block's copy and path pointers in flight
// while this one is computed.
// Inside a segment the taps of token x are x-3 .. x, all in the tile: a
// thread unpacks the 7 rows of its 4 tokens' taps once and slides over them;
// a tap is read again only where the path turns (a segment's first tokens,
// whose taps lie in the parent).  The taps are summed in order 0..3 with
// two-lane float multiply-adds.
constexpr int kConvTok = 128;                     // tokens per block
constexpr int kConvRows = kConvTok + 3;
constexpr int kConvBuf = kConvRows * kGd * 2;   // one block's rows, bf16
constexpr int kConvSmem = 2 * kConvBuf + 128;   // two blocks, 128-byte aligned

__global__ void __launch_bounds__(kConvThreads, kConvPerSm) gdn_conv_kernel(const __grid_constant__ CUtensorMap mx,
                                                                   const GdnParams p, int S) {
  extern __shared__ uint8_t conv_dyn[];
  uint8_t* const xs0 = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(conv_dyn) + 127) & ~uintptr_t(127));
  auto xs = [&](int b) { return xs0 + b * kConvBuf; };   // [kConvRows rows][128 channels] bf16, two blocks
  __shared__ int taps[2][kConvTok][3];   // the 1, 2 and 3 tokens back on each token's path (-2: pad or past the end)
  __shared__ uint32_t plain[2][kConvTok / 32];   // bit t: token t of the block has taps t-3 .. t (no pad, no turn)
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ int abort_flag;
  const int G = 3 * p.H, nbx = (p.N + kConvTok - 1) / kConvTok;
  const int grp = blockIdx.x % G, bx0 = blockIdx.x / G;
  const int lt = threadIdx.x >> 4, vec = threadIdx.x & 15;
  const int ch = grp * kGd + vec * 8;
  const bool is_qk = grp < 2 * p.H;
  auto load_taps = [&](int bx, int& t0, int& t1, int& t2) {
    const int x = bx * kConvTok + threadIdx.x;
    const bool in = x < p.N;
    t0 = in ? p.prev[x] : -2;
    t1 = in ? p.prev2[x] : -1;
    t2 = in ? p.prev3[x] : -1;
  };
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    abort_flag = 0;
    fence_mbar_init();
    if (bx0 < nbx) {
      mbar_expect_tx(&bars[0], kConvBuf);
      tma_load_2d_g(xs(0), &mx, &bars[0], grp * kGd, bx0 * kConvTok - 3);
    }
  }
  // whole warps (a token each) store a block's pointers and plain bits
  auto store_taps = [&](int b, int bx, int t0, int t1, int t2) {
    const int x = bx * kConvTok + threadIdx.x;
    taps[b][threadIdx.x][0] = t0;
    taps[b][threadIdx.x][1] = t1;
    taps[b][threadIdx.x][2] = t2;
    const uint32_t m = __ballot_sync(0xffffffffu, x >= 3 && t0 == x - 1 && t1 == x - 2 && t2 == x - 3);
    if ((threadIdx.x & 31) == 0) plain[b][threadIdx.x >> 5] = m;
  };
  if (threadIdx.x < kConvTok && bx0 < nbx) {
    int t0, t1, t2;
    load_taps(bx0, t0, t1, t2);
    store_taps(0, bx0, t0, t1, t2);
  }
  float2 wt[4][4];   // tap t of channels ch + 2i, ch + 2i + 1
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 w0 = reinterpret_cast<const float4*>(p.conv_w)[ch + 2 * i];
    const float4 w1 = reinterpret_cast<const float4*>(p.conv_w)[ch + 2 * i + 1];
    wt[0][i] = make_float2(w0.x, w1.x);
    wt[1][i] = make_float2(w0.y, w1.y);
    wt[2][i] = make_float2(w0.z, w1.z);
    wt[3][i] = make_float2(w0.w, w1.w);
  }
  // A row's pads are its tail, so a block that lies in one row and starts
  // with a pad is all pads: its rows are not copied (thread 0 reads the
  // block's first pointer one block ahead).
  auto all_pads = [&](int b, int first_prev) {
    const int x0 = b * kConvTok, x1 = min(x0 + kConvTok - 1, p.N - 1);
    return first_prev == -2 && x0 / p.T == x1 / p.T;
  };
  int prev_ahead = (threadIdx.x == 0 && bx0 + S < nbx) ? p.prev[(bx0 + S) * kConvTok] : 0;
  __syncthreads();
  int j = 0;
  for (int bx = bx0; bx < nbx; bx += S, ++j) {
    const int buf = j & 1, nb = bx + S;
    int n0 = -2, n1 = -1, n2 = -1;
    if (nb < nbx) {   // the next block: its rows by TMA (that buffer was freed by the barrier
                      // that ended the previous block), its path pointers into registers
      if (threadIdx.x == 0) {
        if (all_pads(nb, prev_ahead)) {
          mbar_arrive(&bars[buf ^ 1]);   // nothing to copy: complete the phase
        } else {
          mbar_expect_tx(&bars[buf ^ 1], kConvBuf);
          tma_load_2d_g(xs(buf ^ 1), &mx, &bars[buf ^ 1], grp * kGd, nb * kConvTok - 3);
        }
        prev_ahead = nb + S < nbx ? p.prev[(nb + S) * kConvTok] : 0;
      }
      if (threadIdx.x < kConvTok) load_taps(nb, n0, n1, n2);
    }
    if (!__syncthreads_and(mbar_wait(&bars[buf], (j >> 1) & 1, &abort_flag, p.err))) {
      // gave up: let the copies in flight land, then leave
      mbar_wait_drain(&bars[buf], (j >> 1) & 1);
      if (nb < nbx) mbar_wait_drain(&bars[buf ^ 1], ((j + 1) >> 1) & 1);
      return;
    }
    const int xb = bx * kConvTok;
    const uint8_t* xt = xs(buf) + vec * 16;
    // This thread's tokens are xb + tb .. xb + tb + 3 for tb = 4 lt, 64 + 4 lt,
    // ...; tile row r holds token xb - 3 + r, so their in-segment taps are
    // tile rows tb .. tb + 6, each unpacked once into a ring of four rows
    // (row tb + j in win[j & 3]).
#pragma unroll 1
    for (int h = 0; h < kConvTok / 64; ++h) {
      const int tb = 64 * h + 4 * lt;
      const unsigned grpmask = 0xffffu << (threadIdx.x & 16);
      if (((plain[buf][tb >> 5] >> (tb & 31)) & 0xFu) == 0xFu) {
        // The common case, four tokens inside one segment: straight-line code,
        // so the four tokens' chains overlap.  Tile row tb + r is tap r - k of
        // token k; rows are taken in order, so each token sums taps 0..3 in order.
        float2 acc[4][4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[k][i] = make_float2(0.f, 0.f);
#pragma unroll
        for (int r = 0; r < 7; ++r) {
          float f[8];
          unpack8(*reinterpret_cast<const uint4*>(xt + (tb + r) * (kGd * 2)), f);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            if (r - k < 0 || r - k > 3) continue;
#pragma unroll
            for (int i = 0; i < 4; ++i)
              acc[k][i] = __ffma2_rn(wt[r - k][i], make_float2(f[2 * i], f[2 * i + 1]), acc[k][i]);
          }
        }
        float a[4][8];
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            a[k][2 * i] = __fdividef(acc[k][i].x, 1.f + __expf(-acc[k][i].x));
            a[k][2 * i + 1] = __fdividef(acc[k][i].y, 1.f + __expf(-acc[k][i].y));
          }
        if (is_qk) {
          float ss[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            ss[k] = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) ss[k] = fmaf(a[k][i], a[k][i], ss[k]);
          }
#pragma unroll
          for (int o = 8; o >= 1; o >>= 1)
#pragma unroll
            for (int k = 0; k < 4; ++k) ss[k] += __shfl_xor_sync(grpmask, ss[k], o);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float rn = rsqrtf(ss[k] + 1e-6f);
#pragma unroll
            for (int i = 0; i < 8; ++i) a[k][i] *= rn;
          }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint4 out;
          out.x = pack_bf16x2(a[k][0], a[k][1]);
          out.y = pack_bf16x2(a[k][2], a[k][3]);
          out.z = pack_bf16x2(a[k][4], a[k][5]);
          out.w = pack_bf16x2(a[k][6], a[k][7]);
          *reinterpret_cast<uint4*>(p.y + (size_t)(xb + tb + k) * p.C + ch) = out;
        }
      } else {
        float win[4][8];
#pragma unroll
        for (int j = 0; j < 3; ++j) unpack8(*reinterpret_cast<const uint4*>(xt + (tb + j) * (kGd * 2)), win[j]);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int tl = tb + k, x = xb + tl;
          unpack8(*reinterpret_cast<const uint4*>(xt + (tl + 3) * (kGd * 2)), win[(k + 3) & 3]);
          const int p1 = taps[buf][tl][0];
          if (p1 == -2) {
            if (x < p.N && grp < p.H) {   // a pad: o = 0 for head grp
              float4* o4 = reinterpret_cast<float4*>(p.o + ((size_t)x * p.H + grp) * kGd + vec * 8);
              o4[0] = o4[1] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            continue;   // all 16 lanes of a token take the same branch
          }
          const int src[3] = {taps[buf][tl][2], taps[buf][tl][1], p1};   // taps 0..2; tap 3 is x itself
          float2 acc[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[i] = make_float2(0.f, 0.f);
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const float* f = win[(k + t) & 3];
            float g[8];
            if (t < 3 && src[t] != x - 3 + t) {   // the path turns here (or has no such tap)
              if (src[t] < 0) continue;
              const int r = src[t] - (xb - 3);
              const uint4 v = (r >= 0 && r < kConvRows)
                                  ? *reinterpret_cast<const uint4*>(xt + r * (kGd * 2))
                                  : *reinterpret_cast<const uint4*>(p.x + (size_t)src[t] * p.C + ch);
              unpack8(v, g);
              f = g;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[i] = __ffma2_rn(wt[t][i], make_float2(f[2 * i], f[2 * i + 1]), acc[i]);
          }
          float a[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            a[2 * i] = __fdividef(acc[i].x, 1.f + __expf(-acc[i].x));
            a[2 * i + 1] = __fdividef(acc[i].y, 1.f + __expf(-acc[i].y));
          }
          if (is_qk) {
            float ss = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) ss = fmaf(a[i], a[i], ss);
            ss += __shfl_xor_sync(grpmask, ss, 8);
            ss += __shfl_xor_sync(grpmask, ss, 4);
            ss += __shfl_xor_sync(grpmask, ss, 2);
            ss += __shfl_xor_sync(grpmask, ss, 1);
            const float r = rsqrtf(ss + 1e-6f);
#pragma unroll
            for (int i = 0; i < 8; ++i) a[i] *= r;
          }
          uint4 out;
          out.x = pack_bf16x2(a[0], a[1]);
          out.y = pack_bf16x2(a[2], a[3]);
          out.z = pack_bf16x2(a[4], a[5]);
          out.w = pack_bf16x2(a[6], a[7]);
          *reinterpret_cast<uint4*>(p.y + (size_t)x * p.C + ch) = out;
        }
      }
    }
    if (threadIdx.x < kConvTok && nb < nbx) store_taps(buf ^ 1, nb, n0, n1, n2);
    __syncthreads();   // this block's rows and pointers are read; the next block's pointers are in
  }
}

// ---------------------------------------------------------------------------
// Per (chunk, head): everything of the chunk that does not depend on a state.
// [Q K^T; K K^T] is one tcgen05 pass (M = 128, N = 64, K = 128) into TMEM; the
// inverse of the unit-lower-triangular I + A runs on the CUDA cores in
// float32, and its products with V and K are two more tcgen05 passes
// (M = 128, N = 128, K = 64, hi and lo halves of T accumulated).

__global__ void __launch_bounds__(kPrepThreads, 2) gdn_prep_kernel(const GdnParams p) {
  extern __shared__ uint8_t prep_dyn[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(prep_dyn) + 1023) & ~uintptr_t(1023));
  uint8_t* tile = sm;                                              // [Q; K]
  uint8_t* sv = sm + kPoV;                                         // V, MN-major operand
  float* sA = reinterpret_cast<float*>(sm + kPoA);                 // [64 columns][68]
  uint8_t* sT = sm + kPoT;                                         // [T'; T''] hi, then lo
  float* sgam = reinterpret_cast<float*>(sm + kPoGam);
  float* sbeta = reinterpret_cast<float*>(sm + kPoBeta);
  float* seg = reinterpret_cast<float*>(sm + kPoEg);               // e^{gam_t}
  float* sek = reinterpret_cast<float*>(sm + kPoEk);               // e^{gam_L - gam_t}
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + kPoBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ch = p.chunk0 + (int)(blockIdx.x / p.H), h = blockIdx.x % p.H;
  const int x0 = p.chunk_start[ch], L = p.chunk_len[ch];
  const int Hd = p.H * kGd;
  const size_t row = (size_t)ch * p.H + h;

  if (tid == 0) {
    mbar_init(bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  {   // all twelve 16-byte loads of a thread in flight before any is stored
    constexpr int kIt = kGc * 16 / kPrepThreads;
    uint4 rq[kIt], rk[kIt], rv[kIt];
#pragma unroll
    for (int u = 0; u < kIt; ++u) {
      const int i = tid + u * kPrepThreads, t = i >> 4, c = (i & 15) * 8;
      rq[u] = rk[u] = rv[u] = make_uint4(0, 0, 0, 0);
      if (t < L) {
        const __nv_bfloat16* yr = p.y + (size_t)(x0 + t) * p.C + h * kGd + c;
        rq[u] = *reinterpret_cast<const uint4*>(yr);
        rk[u] = *reinterpret_cast<const uint4*>(yr + Hd);
        rv[u] = *reinterpret_cast<const uint4*>(yr + 2 * Hd);
      }
    }
#pragma unroll
    for (int u = 0; u < kIt; ++u) {
      const int i = tid + u * kPrepThreads, t = i >> 4, c = (i & 15) * 8;
      const int off = (c >> 6) * 16384 + ((((c & 63) >> 3) ^ (t & 7)) << 4);
      *reinterpret_cast<uint4*>(tile + off + t * 128) = rq[u];
      *reinterpret_cast<uint4*>(tile + off + (kGc + t) * 128) = rk[u];
      *reinterpret_cast<uint4*>(sv + (c >> 6) * 8192 + t * 128 + ((((c & 63) >> 3) ^ (t & 7)) << 4)) = rv[u];
    }
  }
  if (tid < kGc) {
    sgam[tid] = tid < L ? p.g[(size_t)(x0 + tid) * p.H + h] : 0.f;
    sbeta[tid] = tid < L ? p.beta[(size_t)(x0 + tid) * p.H + h] : 0.f;
  }
  fence_proxy_async_smem();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  if (tid == 0) {
    constexpr uint32_t idesc = idesc_bf16(128, 64, 0, 0);
    const uint32_t tb = smem_u32(tile);
#pragma unroll
    for (int s = 0; s < 8; ++s)
      mma_ss_lo(tmem, desc_lo_kmajor(tb + (s >> 2) * 16384 + (s & 3) * 32),
                desc_lo_kmajor(tb + (s >> 2) * 16384 + 8192 + (s & 3) * 32), idesc, s > 0 ? 1u : 0u);
    mma_commit(bar);
  }
  if (tid < 32) {   // inclusive prefix sum of g over the 64 rows, and the row exponentials
    float a = sgam[tid], b = sgam[tid + 32];
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
    sgam[tid] = a;
    sgam[tid + 32] = b;
    seg[tid] = expf(a);
    seg[tid + 32] = expf(b);
    sek[tid] = expf(gl - a);
    sek[tid + 32] = expf(gl - b);
  }
  __syncthreads();

  // A (strictly lower, from K K^T) and P (lower with the diagonal, from Q K^T):
  // warp w reads TMEM rows 32 (w % 4) .. + 31, columns 32 (w / 4) .. + 31
  {
    const bool ready = mbar_wait(bar, 0, abort_flag, p.err);
    fence_after_sync();
    uint32_t v[32];
    const int m = 32 * (warp & 3) + lane, j0 = 32 * (warp >> 2);
    tmem_ld32(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + j0, v);
    tmem_ld_wait();
    if (m < kGc) {
      const int i = m;
      const float gi = sgam[i];
      uint32_t pw[16];
#pragma unroll
      for (int q = 0; q < 32; q += 2) {
        float f[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int j = j0 + q + e;
          f[e] = (ready && j <= i && i < L) ? p.scale * __expf(gi - sgam[j]) * __uint_as_float(v[q + e]) : 0.f;
        }
        pw[q / 2] = pack_bf16x2(f[0], f[1]);
      }
      uint4* dst = reinterpret_cast<uint4*>(p.pm + (row * kGc + i) * kGc + j0);
#pragma unroll
      for (int q = 0; q < 4; ++q) dst[q] = make_uint4(pw[4 * q], pw[4 * q + 1], pw[4 * q + 2], pw[4 * q + 3]);
    } else {
      const int i = m - kGc;
      const float gi = sgam[i], bi = sbeta[i];
#pragma unroll
      for (int q = 0; q < 32; ++q) {
        const int j = j0 + q;
        sA[j * kPrepLa + i] = (ready && j < i) ? bi * __expf(gi - sgam[j]) * __uint_as_float(v[q]) : 0.f;
      }
    }
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();

  // Q~ (rows 0..63 of the [Q~; W] tile) and K~, 8 channels (16 bytes) per item
  for (int it = tid; it < 2 * kGc * 16; it += kPrepThreads) {
    const int m = it >> 4, c = (it & 15) * 8, t = m & (kGc - 1);   // m < 64: a Q row, else a K row
    const float sc = t < L ? (m < kGc ? p.scale * seg[t] : sek[t]) : 0.f;
    const uint4 r = *reinterpret_cast<const uint4*>(tile + (c >> 6) * 16384 + m * 128 +
                                                    ((((c & 63) >> 3) ^ (m & 7)) << 4));
    float f[8];
    unpack8(r, f);
    const uint4 o = make_uint4(pack_bf16x2(sc * f[0], sc * f[1]), pack_bf16x2(sc * f[2], sc * f[3]),
                               pack_bf16x2(sc * f[4], sc * f[5]), pack_bf16x2(sc * f[6], sc * f[7]));
    __nv_bfloat16* dst = m < kGc ? p.wq + (row * 128 + t) * kGd + c : p.kt + (row * kGc + t) * kGd + c;
    *reinterpret_cast<uint4*>(dst) = o;
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();

  // T = (I + A)^{-1} in 32 x 32 blocks: T11 = (I + A11)^{-1} and
  // T22 = (I + A22)^{-1} (one warp each, a column per thread, column-oriented
  // substitution: once an entry is final it is taken out of every later
  // row), then T21 = -T22 (A21 T11).  T is kept float32 row-major [64][64]
  // over the Q rows of the tile (read above): rows 0-31 in the first 8 KB
  // half, rows 32-63 in the second; A21 T11 goes over A22's columns of A.
  auto trow = [&](int t) { return reinterpret_cast<float*>(tile + (t >> 5) * 16384 + (t & 31) * 256); };
  float* sM = sA + 32 * kPrepLa;   // [32][32] row-major
  if (warp < 2) {
    const int b0 = 32 * warp, cc = b0 + lane;   // block rows / columns b0 .. b0 + 31; this thread's column
    float x[32];
#pragma unroll
    for (int t = 0; t < 32; ++t) x[t] = t == lane ? 1.f : 0.f;
#pragma unroll
    for (int t = 0; t < 31; ++t) {
      const float xt = x[t];
#pragma unroll
      for (int r4 = ((t + 1) & ~3); r4 < 32; r4 += 4) {
        const float4 a = *reinterpret_cast<const float4*>(sA + (b0 + t) * kPrepLa + b0 + r4);
        x[r4] = fmaf(-a.x, xt, x[r4]);
        x[r4 + 1] = fmaf(-a.y, xt, x[r4 + 1]);
        x[r4 + 2] = fmaf(-a.z, xt, x[r4 + 2]);
        x[r4 + 3] = fmaf(-a.w, xt, x[r4 + 3]);
      }
    }
#pragma unroll
    for (int t = 0; t < 32; ++t) trow(b0 + t)[cc] = x[t];
  } else {
    for (int it = tid - 64; it < 32 * 32; it += kPrepThreads - 64) trow(it >> 5)[32 + (it & 31)] = 0.f;   // T12
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  {   // M = A21 T11: thread = (row r, columns 4 c4 .. + 3)
    const int r = tid >> 3, c4 = (tid & 7) * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int k = 0; k < 32; ++k) {
      const float a = sA[k * kPrepLa + 32 + r];
      const float4 tv = *reinterpret_cast<const float4*>(trow(k) + c4);
      acc.x = fmaf(a, tv.x, acc.x);
      acc.y = fmaf(a, tv.y, acc.y);
      acc.z = fmaf(a, tv.z, acc.z);
      acc.w = fmaf(a, tv.w, acc.w);
    }
    *reinterpret_cast<float4*>(sM + r * 32 + c4) = acc;   // A22 was last read before the barrier above
  }
  __syncthreads();
  {   // T21 = -T22 M
    const int r = tid >> 3, c4 = (tid & 7) * 4;
    const float* t22 = trow(32 + r) + 32;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int k = 0; k < 32; ++k) {
      const float a = t22[k];
      const float4 mv = *reinterpret_cast<const float4*>(sM + k * 32 + c4);
      acc.x = fmaf(a, mv.x, acc.x);
      acc.y = fmaf(a, mv.y, acc.y);
      acc.z = fmaf(a, mv.z, acc.z);
      acc.w = fmaf(a, mv.w, acc.w);
    }
    *reinterpret_cast<float4*>(trow(32 + r) + c4) = make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
  }
  __syncthreads();
  // T' = T diag(beta) and T'' = T diag(beta e^gam), split into bf16 hi + lo,
  // to the operand tiles (rows 0-63 T', rows 64-127 T'', K index s); an item
  // is one 16-byte chunk (8 columns) of one row
  for (int it = tid; it < kGc * 8; it += kPrepThreads) {
    const int t = it >> 3, s0 = (it & 7) * 8;
    const float* tr = trow(t) + s0;
    float f[8];
    *reinterpret_cast<float4*>(f) = *reinterpret_cast<const float4*>(tr);
    *reinterpret_cast<float4*>(f + 4) = *reinterpret_cast<const float4*>(tr + 4);
#pragma unroll
    for (int part = 0; part < 2; ++part) {
      uint32_t hw[4], lw[4];
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        float v[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int sc = s0 + e + q;
          v[q] = f[e + q] * (part ? sbeta[sc] * seg[sc] : sbeta[sc]);
        }
        const __nv_bfloat162 h2 = __floats2bfloat162_rn(v[0], v[1]);
        const float2 hf = __bfloat1622float2(h2);
        const __nv_bfloat162 l2 = __floats2bfloat162_rn(v[0] - hf.x, v[1] - hf.y);
        hw[e / 2] = *reinterpret_cast<const uint32_t*>(&h2);
        lw[e / 2] = *reinterpret_cast<const uint32_t*>(&l2);
      }
      const int m = part * kGc + t;
      const int off = m * 128 + (((s0 >> 3) ^ (m & 7)) << 4);
      *reinterpret_cast<uint4*>(sT + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      *reinterpret_cast<uint4*>(sT + 16384 + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
  }
  fence_proxy_async_smem();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  // [T'; T''] (hi + lo) x V into columns 0-127 (rows 0-63: U^ = T' V) and
  // x K into columns 128-255 (rows 64-127: W = T'' K); the [Q K^T; K K^T]
  // accumulator in columns 0-63 was read above.
  if (tid == 0) {
    constexpr uint32_t idesc = idesc_bf16(128, 128, 0, 1);
    const uint32_t ta = smem_u32(sT), tv = smem_u32(sv), tk = smem_u32(tile) + 8192;
#pragma unroll
    for (int hl = 0; hl < 2; ++hl)
#pragma unroll
      for (int s4 = 0; s4 < 4; ++s4) {
        const uint32_t a = desc_lo_kmajor(ta + hl * 16384 + s4 * 32);
        mma_ss_lo(tmem, a, desc_lo_mn8k(tv + s4 * 2048), idesc, (hl | s4) ? 1u : 0u);
        mma_ss_lo(tmem + 128, a, desc_lo_mn16k(tk + s4 * 2048), idesc, (hl | s4) ? 1u : 0u);
      }
    mma_commit(bar);
  }
  {
    const bool ready = mbar_wait(bar, 1, abort_flag, p.err);
    fence_after_sync();
    // warp w reads TMEM rows 32 (w % 4) .. + 31 (thread = row), columns half (w / 4) of 64
    const int q4 = warp & 3, half = warp >> 2, m = 32 * q4 + lane;
    const uint32_t lrow = (uint32_t)(32 * q4) << 16;
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      uint32_t v[32];
      const int d0 = half * 64 + cc * 32;
      tmem_ld32(tmem + lrow + (q4 < 2 ? 0 : 128) + d0, v);
      tmem_ld_wait();
      if (!ready) continue;
      if (q4 < 2) {   // U^ transposed: [d][t], a warp writes 128 contiguous bytes per d
        float* dst = p.ut + (row * kGd + d0) * kGc + m;
#pragma unroll
        for (int j = 0; j < 32; ++j) dst[(size_t)j * kGc] = __uint_as_float(v[j]);
      } else {        // W: bf16 rows 64..127 of the [Q~; W] tile
        uint4* dst = reinterpret_cast<uint4*>(p.wq + (row * 128 + m) * kGd + d0);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          dst[j] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * j]), __uint_as_float(v[8 * j + 1])),
                              pack_bf16x2(__uint_as_float(v[8 * j + 2]), __uint_as_float(v[8 * j + 3])),
                              pack_bf16x2(__uint_as_float(v[8 * j + 4]), __uint_as_float(v[8 * j + 5])),
                              pack_bf16x2(__uint_as_float(v[8 * j + 6]), __uint_as_float(v[8 * j + 7])));
      }
    }
  }
  if (tid == 0) p.decay[row] = expf(sgam[L - 1]);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

// ---------------------------------------------------------------------------
// One CTA per (segment of this depth, head).  Per chunk i the critical chain is
// E1(i) -> [Q~; W] S0 -> V'(i) -> P V', K~^T V' -> E1(i + 1); the output rows
// of chunk i - 1 leave (through padded shared memory and one bulk copy per
// row) while the tensor core works on chunk i, from the other of two
// accumulator buffers.
__global__ void __launch_bounds__(kStThreads, 1)
    gdn_state_kernel(const __grid_constant__ CUtensorMap mwq, const __grid_constant__ CUtensorMap mkt,
                     const __grid_constant__ CUtensorMap mpm, const GdnParams p) {
  extern __shared__ uint8_t gsm_dyn[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(gsm_dyn) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + B_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const float* ut_s = reinterpret_cast<const float*>(sm + kOffUt);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sidx = p.seg0 + (int)(blockIdx.x / p.H), h = (int)(blockIdx.x % p.H);
  const int c0 = p.seg_chunk0[sidx], nck = (p.seg_len[sidx] + kGc - 1) / kGc;
  const int par = p.seg_parent[sidx];

  if (threadIdx.x == 0) {
    for (int b = 0; b < B_COUNT; ++b) mbar_init(&bars[b], (b == B_SR || b == B_VR) ? 8 : (b == B_UE) ? 4 : 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  // columns 0-127: the state S; 128 + 128 b (b = chunk parity): [Q~ S0 + P V' ; W S0]
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    if (lane == 0) {
      // ------------------------------------------------------------ loads
      tma_prefetch_desc(&mwq);
      tma_prefetch_desc(&mkt);
      tma_prefetch_desc(&mpm);
      int lastf[2] = {-1, -1}, lastu = -1;
      for (int i = 0; i < nck; ++i) {
        const int st = i & 1;
        if (i >= 2 && !mbar_wait(&bars[B_E + st], ((i >> 1) - 1) & 1, abort_flag, p.err)) break;
        const int row = (c0 + i) * p.H + h;
        uint8_t* stage = sm + st * kStStage;
        mbar_expect_tx(&bars[B_F + st], 32768 + 16384 + 8192);
        tma_load_2d_g(stage, &mwq, &bars[B_F + st], 0, row * 128);
        tma_load_2d_g(stage + 16384, &mwq, &bars[B_F + st], 64, row * 128);
        tma_load_2d_g(stage + kOffKt, &mkt, &bars[B_F + st], 0, row * kGc);
        tma_load_2d_g(stage + kOffKt + 8192, &mkt, &bars[B_F + st], 64, row * kGc);
        tma_load_2d_g(stage + kOffP, &mpm, &bars[B_F + st], 0, row * kGc);
        lastf[st] = (i >> 1) & 1;
        if (i >= 1 && !mbar_wait(&bars[B_UE], (i - 1) & 1, abort_flag, p.err)) break;
        mbar_expect_tx(&bars[B_UF], 32768);
        bulk_load(sm + kOffUt, p.ut + (size_t)row * kGd * kGc, 32768, &bars[B_UF]);
        lastu = i & 1;
      }
      for (int st = 0; st < 2; ++st)
        if (lastf[st] >= 0) mbar_wait_drain(&bars[B_F + st], lastf[st]);
      if (lastu >= 0) mbar_wait_drain(&bars[B_UF], lastu);
    }
    __syncwarp();
  } else if (warp == 9) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA
      constexpr uint32_t id_kmn = idesc_bf16(128, 128, 0, 1);
      constexpr uint32_t id_mnmn = idesc_bf16(128, 128, 1, 1);
      for (int i = 0; i < nck; ++i) {
        const int st = i & 1;
        const uint32_t stage = sb + st * kStStage, d1 = tmem + 128 + 128 * (i & 1);
        if (!mbar_wait(&bars[B_SR], i & 1, abort_flag, p.err)) break;
        if (!mbar_wait(&bars[B_F + st], (i >> 1) & 1, abort_flag, p.err)) break;
        fence_after_sync();
        // [Q~; W] S0
#pragma unroll
        for (int s = 0; s < 8; ++s)
          mma_ss_lo(d1, desc_lo_kmajor(stage + (s >> 2) * 16384 + (s & 3) * 32),
                    desc_lo_mnmajor(sb + kOffSop + s * 2048), id_kmn, s > 0 ? 1u : 0u);
        mma_commit(&bars[B_M1]);
        if (!mbar_wait(&bars[B_VR], i & 1, abort_flag, p.err)) break;
        fence_after_sync();
        // rows 0-63: Q~ S0 + P V';  state: e^{gam_L} S0 + K~^T V'
#pragma unroll
        for (int s = 0; s < 4; ++s)
          mma_ss_lo(d1, desc_lo_kmajor(stage + kOffP + s * 32), desc_lo_mn8k(sb + kOffVop + s * 2048), id_kmn, 1u);
#pragma unroll
        for (int s = 0; s < 4; ++s)
          mma_ss_lo(tmem, desc_lo_mn8k(stage + kOffKt + s * 2048), desc_lo_mn8k(sb + kOffVop + s * 2048), id_mnmn,
                    1u);
        mma_commit(&bars[B_M2]);
        mma_commit(&bars[B_E + st]);
      }
      mma_commit(&bars[B_DRAIN]);
      mbar_wait_drain(&bars[B_DRAIN], 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // thread = (TMEM lane r, column half hc): warps w and w + 4 share lanes 32 (w % 4) ..
    const int r = threadIdx.x & 127, hc = warp >> 2;   // r: the state's k row; of the accumulator, the chunk row
    const uint32_t lrow = (uint32_t)((warp & 3) * 32) << 16, col0 = (uint32_t)hc * 64;
    uint32_t v[64];
    // Half of a padded 528-byte row per thread: into shared memory, then one bulk copy to HBM.
    auto row_out = [&](uint8_t* buf, float* dst) {
      bulk_wait_read0();   // the previous copy from this half row has read it
      buf += hc * 256;
#pragma unroll
      for (int q = 0; q < 16; ++q)
        reinterpret_cast<uint4*>(buf)[q] = make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      fence_proxy_async_smem();
      bulk_store(dst + col0, buf, 256);
      bulk_commit();
    };
    {
      const float* src = par >= 0 ? p.state + (((size_t)par * p.H + h) * kGd + r) * kGd + col0 : nullptr;
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {
#pragma unroll
        for (int q = 0; q < 32; ++q) v[q] = src ? __float_as_uint(src[cc * 32 + q]) : 0u;
        tmem_st32(tmem + lrow + col0 + cc * 32, v);
      }
      tmem_st_wait();
    }
    bool ok = true;
    // the chunk's scalars are read one chunk ahead
    int L = p.chunk_len[c0], x0 = p.chunk_start[c0], L_prev = 0, x0_prev = 0;
    float dec = p.decay[c0 * p.H + h];
    for (int i = 0; ok && i < nck; ++i) {
      int L_next = 0, x0_next = 0;
      float dec_next = 0.f;
      if (i + 1 < nck) {
        L_next = p.chunk_len[c0 + i + 1];
        x0_next = p.chunk_start[c0 + i + 1];
        dec_next = p.decay[(c0 + i + 1) * p.H + h];
      }
      // E1: S0 -> bf16 operand (k rows, v contiguous in two 64-column halves: this
      // thread's half is one of them); S <- e^{gam_L} S0
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) tmem_ld32(tmem + lrow + col0 + cc * 32, v + 32 * cc);
      tmem_ld_wait();
      {
        uint8_t* half = sm + kOffSop + hc * 16384 + r * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t* e = v + 8 * j;
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(e[0]), __uint_as_float(e[1]));
          w.y = pack_bf16x2(__uint_as_float(e[2]), __uint_as_float(e[3]));
          w.z = pack_bf16x2(__uint_as_float(e[4]), __uint_as_float(e[5]));
          w.w = pack_bf16x2(__uint_as_float(e[6]), __uint_as_float(e[7]));
          *reinterpret_cast<uint4*>(half + ((j ^ (r & 7)) << 4)) = w;
        }
      }
      fence_proxy_async_smem();
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_SR]);
      // the decayed state goes back while [Q~; W] S0 runs (that product reads
      // the bf16 copy); K~^T V' adds to it only after every warp's B_VR arrival
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t w[32];
#pragma unroll
        for (int q = 0; q < 32; ++q) w[q] = __float_as_uint(__uint_as_float(v[32 * cc + q]) * dec);
        tmem_st32(tmem + lrow + col0 + cc * 32, w);
      }
      tmem_st_wait();
      if ((warp & 3) < 2) {   // the E2 warps arrive once V' is in place too
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[B_VR]);   // this warp's part of the state is stored
      }
      if (p.s0) {   // training: keep the chunk's starting state for the backward, as [d_v][d_k]
                    // (off the chain: the products of this chunk already run)
        float* d = p.s0 + (size_t)((c0 + i) * p.H + h) * kGd * kGd + (size_t)col0 * kGd + r;
#pragma unroll
        for (int q = 0; q < 64; ++q) d[q * kGd] = __uint_as_float(v[q]);
      }

      if ((warp & 3) < 2) {
        // E3 of the previous chunk: its output rows 0-63 of the other accumulator
        if (i > 0) {
          const uint32_t d1p = tmem + 128 + 128 * ((i - 1) & 1);
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) tmem_ld32(d1p + lrow + col0 + cc * 32, v + 32 * cc);
          tmem_ld_wait();
          if (r < L_prev) row_out(sm + kOffOst + r * kOstLd, p.o + ((size_t)(x0_prev + r) * p.H + h) * kGd);
        }
      } else {
        // E2: V' = U^ - W S0 on rows 64-127 (chunk row r - 64)
        const int t = r - 64;
        if (!__all_sync(0xffffffffu, mbar_wait(&bars[B_M1], i & 1, abort_flag, p.err)) ||
            !__all_sync(0xffffffffu, mbar_wait(&bars[B_UF], i & 1, abort_flag, p.err))) {
          ok = false;
          break;
        }
        fence_after_sync();
        const uint32_t d1 = tmem + 128 + 128 * (i & 1);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) tmem_ld32(d1 + lrow + col0 + cc * 32, v + 32 * cc);
        tmem_ld_wait();
        uint8_t* half = sm + kOffVop + hc * 8192 + t * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float f[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int col = 8 * j + e;
            f[e] = ut_s[(col0 + col) * kGc + t] - __uint_as_float(v[col]);
          }
          uint4 w;
          w.x = pack_bf16x2(f[0], f[1]);
          w.y = pack_bf16x2(f[2], f[3]);
          w.z = pack_bf16x2(f[4], f[5]);
          w.w = pack_bf16x2(f[6], f[7]);
          *reinterpret_cast<uint4*>(half + ((j ^ (t & 7)) << 4)) = w;
        }
        fence_proxy_async_smem();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bars[B_VR]);
          mbar_arrive(&bars[B_UE]);
        }
      }
      // the state of the next chunk
      if (!__all_sync(0xffffffffu, mbar_wait(&bars[B_M2], i & 1, abort_flag, p.err))) {
        ok = false;
        break;
      }
      fence_after_sync();
      L_prev = L;
      x0_prev = x0;
      L = L_next;
      x0 = x0_next;
      dec = dec_next;
    }
    if (ok) {
      if ((warp & 3) < 2) {   // the last chunk's output rows
        const uint32_t d1p = tmem + 128 + 128 * ((nck - 1) & 1);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) tmem_ld32(d1p + lrow + col0 + cc * 32, v + 32 * cc);
        tmem_ld_wait();
        if (r < L_prev) row_out(sm + kOffOst + r * kOstLd, p.o + ((size_t)(x0_prev + r) * p.H + h) * kGd);
      }
      // the segment's final state, for its children (rows 64-127 go through the
      // operand buffers, which no MMA reads any more)
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) tmem_ld32(tmem + lrow + col0 + cc * 32, v + 32 * cc);
      tmem_ld_wait();
      uint8_t* buf = r < 64 ? sm + kOffOst + r * kOstLd : sm + kOffSop + (r - 64) * kOstLd;
      row_out(buf, p.state + (((size_t)sidx * p.H + h) * kGd + r) * kGd);
    }
    bulk_wait_all0();
  }

  __syncwarp();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == 9) tmem_dealloc(tmem, 512);
}

}  // namespace
}  // namespace stp

using namespace stp;

namespace {

stp_status ws_size(const stp_gdn_desc* desc, const void* plan, size_t* ws_bytes, bool train) {
  clear_error();
  stp_status st = check_gdn_desc(desc);
  if (st) return st;
  const int32_t* w = static_cast<const int32_t*>(plan);
  if ((st = check_gdn_plan(desc, w))) return st;
  if (!ws_bytes) return fail(STP_EINVAL, "stp_gdn_workspace_size: NULL output");
  const GdnLayout L = gdn_layout(w[GP_N], desc->n_heads, w[GP_NCHUNK], w[GP_NSEG]);
  *ws_bytes = train ? L.train_total : L.total;
  return STP_OK;
}

// Two library streams per device for the forward: "hi" (the greatest
// priority) prepares the chunks of depth 0 and runs their state walk, "aux"
// prepares the other depths' chunks meanwhile.
struct GdnStreams {
  bool ready = false;
  cudaStream_t hi = nullptr, aux = nullptr;
  cudaEvent_t fork = nullptr, join_hi = nullptr, join_aux = nullptr, dep1 = nullptr;
};
std::mutex g_gdn_mu;
GdnStreams g_gdn_streams[64];

cudaError_t gdn_streams(GdnStreams** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_gdn_mu);
  GdnStreams& g = g_gdn_streams[dev];
  if (!g.ready) {
    int least = 0, greatest = 0;
    e = cudaDeviceGetStreamPriorityRange(&least, &greatest);
    if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&g.hi, cudaStreamNonBlocking, greatest);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&g.aux, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&g.fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&g.join_hi, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&g.join_aux, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&g.dep1, cudaEventDisableTiming);
    if (e != cudaSuccess) return e;
    g.ready = true;
  }
  *out = &g;
  return cudaSuccess;
}

stp_status gdn_forward(const stp_gdn_desc* desc, const void* plan, const void* d_plan, const void* x,
                       const float* conv_w, const float* g, const float* beta, float* o, void* d_ws, void* stream,
                       bool train) {
  clear_error();
  stp_status st = check_gdn_desc(desc);
  if (st) return st;
  const int32_t* w = static_cast<const int32_t*>(plan);
  if ((st = check_gdn_plan(desc, w))) return st;
  if (!d_plan || !x || !conv_w || !g || !beta || !o || !d_ws)
    return fail(STP_EINVAL, "stp_gdn_fwd: NULL device pointer");
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(conv_w) | reinterpret_cast<uintptr_t>(o)) & 15 ||
      (reinterpret_cast<uintptr_t>(d_ws) | reinterpret_cast<uintptr_t>(d_plan)) & 255)
    return fail(STP_EINVAL, "stp_gdn_fwd: x, conv_w, o 16-byte, d_plan and ws 256-byte aligned");
  const int N = w[GP_N], H = desc->n_heads, n_chunk = w[GP_NCHUNK], n_seg = w[GP_NSEG], n_depth = w[GP_NDEPTH];
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (N == 0) {
    // nothing to compute, but the error word still starts this call cleared
    const cudaError_t e0 = cudaMemsetAsync(d_ws, 0, 4, s);
    return e0 == cudaSuccess ? STP_OK : fail(STP_ECUDA, "stp_gdn_fwd: %s", cudaGetErrorString(e0));
  }
  const int32_t* dp = static_cast<const int32_t*>(d_plan);
  GdnParams p;
  p.N = N;
  p.T = desc->row_len;
  p.H = H;
  p.C = 3 * H * kGd;
  p.seg0 = 0;
  p.chunk0 = 0;
  p.scale = desc->scale;
  p.prev = dp + w[GP_PREV];
  p.prev2 = dp + w[GP_PREV2];
  p.prev3 = dp + w[GP_PREV3];
  p.seg_len = dp + w[GP_SEG_LEN];
  p.seg_parent = dp + w[GP_SEG_PARENT];
  p.seg_chunk0 = dp + w[GP_SEG_CHUNK0];
  p.chunk_start = dp + w[GP_CHUNK_START];
  p.chunk_len = dp + w[GP_CHUNK_LEN];
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.conv_w = conv_w;
  p.g = g;
  p.beta = beta;
  char* ws = static_cast<char*>(d_ws);
  const GdnLayout L = gdn_layout(N, H, n_chunk, n_seg);
  p.err = reinterpret_cast<uint32_t*>(ws);
  p.y = reinterpret_cast<__nv_bfloat16*>(ws + L.y);
  p.wq = reinterpret_cast<__nv_bfloat16*>(ws + L.wq);
  p.kt = reinterpret_cast<__nv_bfloat16*>(ws + L.kt);
  p.pm = reinterpret_cast<__nv_bfloat16*>(ws + L.pm);
  p.ut = reinterpret_cast<float*>(ws + L.ut);
  p.decay = reinterpret_cast<float*>(ws + L.decay);
  p.state = reinterpret_cast<float*>(ws + L.state);
  p.s0 = train ? reinterpret_cast<float*>(ws + L.s0) : nullptr;
  p.o = o;
  CUtensorMap mwq, mkt, mpm, mx;
  if (N > 0 && !make_map_x(&mx, p.x, N, (int)p.C, kConvRows))
    return fail(STP_ECUDA, "stp_gdn_fwd: tensor map encoding failed");
  if (n_chunk > 0 &&
      (!make_map_2d(&mwq, p.wq, (int64_t)n_chunk * H * 128, kGd, 128) ||
       !make_map_2d(&mkt, p.kt, (int64_t)n_chunk * H * kGc, kGd, kGc) ||
       !make_map_2d(&mpm, p.pm, (int64_t)n_chunk * H * kGc, kGc, kGc)))
    return fail(STP_ECUDA, "stp_gdn_fwd: tensor map encoding failed");
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(gdn_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPrepSmem);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(gdn_conv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kConvSmem);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(gdn_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kStSmem);
  });
  cudaError_t e = attr_err;
  if (e == cudaSuccess) e = cudaMemsetAsync(p.err, 0, 4, s);
  if (e != cudaSuccess) return fail(STP_ECUDA, "stp_gdn_fwd: %s", cudaGetErrorString(e));
  if (N > 0) {
    // a CTA per (channel group, one of S token-block strides): kConvPerSm resident per SM
    static int n_sm = 0;
    if (n_sm == 0) {
      int dev = 0;
      if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) !=
                                                    cudaSuccess || n_sm <= 0)
        n_sm = 148;
    }
    const int G = 3 * H, nbx = (N + kConvTok - 1) / kConvTok;
    const int S = std::max(1, std::min(nbx, kConvPerSm * n_sm / G));
    gdn_conv_kernel<<<(unsigned)(G * S), kConvThreads, kConvSmem, s>>>(mx, p, S);
  }
  // The chunks of depth 0 are prepared and every depth is walked on a
  // high-priority stream (a walk is one CTA per head and segment: a few SMs),
  // while a second stream prepares the depth-1 chunks, then the deeper ones;
  // the depth-1 walk waits for the first of those, the deeper walks for
  // both.  Chunks are numbered depth by depth.
  const int32_t* depth_off = w + w[GP_DEPTH_OFF];
  const int32_t* seg_chunk0 = w + w[GP_SEG_CHUNK0];
  const int c1 = n_depth > 1 ? seg_chunk0[depth_off[1]] : n_chunk;   // first chunk below depth 0
  const int c2 = n_depth > 2 ? seg_chunk0[depth_off[2]] : n_chunk;   // first chunk below depth 1
  auto walk = [&](int d, cudaStream_t st) {
    const int n = depth_off[d + 1] - depth_off[d];
    if (n <= 0) return;
    GdnParams q = p;
    q.seg0 = depth_off[d];
    gdn_state_kernel<<<(unsigned)(n * H), kStThreads, kStSmem, st>>>(mwq, mkt, mpm, q);
  };
  GdnStreams* gs = nullptr;
  if (c1 < n_chunk) {
    if ((e = gdn_streams(&gs)) != cudaSuccess) return fail(STP_ECUDA, "stp_gdn_fwd: %s", cudaGetErrorString(e));
    std::lock_guard<std::mutex> lock(g_gdn_mu);
    e = cudaEventRecord(gs->fork, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(gs->hi, gs->fork, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(gs->aux, gs->fork, 0);
    if (e == cudaSuccess) {
      if (c1 > 0) gdn_prep_kernel<<<(unsigned)(c1 * H), kPrepThreads, kPrepSmem, gs->hi>>>(p);
      walk(0, gs->hi);
      GdnParams q = p;
      q.chunk0 = c1;
      gdn_prep_kernel<<<(unsigned)((c2 - c1) * H), kPrepThreads, kPrepSmem, gs->aux>>>(q);
      e = cudaEventRecord(gs->dep1, gs->aux);
    }
    if (e == cudaSuccess && c2 < n_chunk) {
      GdnParams q = p;
      q.chunk0 = c2;
      gdn_prep_kernel<<<(unsigned)((n_chunk - c2) * H), kPrepThreads, kPrepSmem, gs->aux>>>(q);
    }
    if (e == cudaSuccess) e = cudaEventRecord(gs->join_aux, gs->aux);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(gs->hi, gs->dep1, 0);
    if (e == cudaSuccess) {
      walk(1, gs->hi);
      e = cudaStreamWaitEvent(gs->hi, gs->join_aux, 0);
    }
    if (e == cudaSuccess) {
      for (int d = 2; d < n_depth; ++d) walk(d, gs->hi);
      e = cudaEventRecord(gs->join_hi, gs->hi);
    }
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, gs->join_hi, 0);
    if (e != cudaSuccess) return fail(STP_ECUDA, "stp_gdn_fwd: %s", cudaGetErrorString(e));
  } else {
    if (n_chunk > 0) gdn_prep_kernel<<<(unsigned)(n_chunk * H), kPrepThreads, kPrepSmem, s>>>(p);
    for (int d = 0; d < n_depth; ++d) walk(d, s);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(STP_ECUDA, "stp_gdn_fwd: %s", cudaGetErrorString(e));
  return STP_OK;
}

}  // namespace

extern "C" stp_status stp_gdn_workspace_size(const stp_gdn_desc* desc, const void* plan, size_t* ws_bytes) {
  return ws_size(desc, plan, ws_bytes, false);
}

extern "C" stp_status stp_gdn_train_workspace_size(const stp_gdn_desc* desc, const void* plan, size_t* ws_bytes) {
  return ws_size(desc, plan, ws_bytes, true);
}

extern "C" stp_status stp_gdn_fwd(const stp_gdn_desc* desc, const void* plan, const void* d_plan, const void* x,
                                  const float* conv_w, const float* g, const float* beta, float* o, void* d_ws,
                                  void* stream) {
  return gdn_forward(desc, plan, d_plan, x, conv_w, g, beta, o, d_ws, stream, false);
}

extern "C" stp_status stp_gdn_fwd_train(const stp_gdn_desc* desc, const void* plan, const void* d_plan,
                                        const void* x, const float* conv_w, const float* g, const float* beta,
                                        float* o, void* d_ws, void* stream) {
  return gdn_forward(desc, plan, d_plan, x, conv_w, g, beta, o, d_ws, stream, true);
}
