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
// Three kernels, float32 on the CUDA cores throughout:
//   gdn_bwd_walk_kernel   one launch per depth, deepest first; one CTA per
//                         (segment, head) walks its chunks last to first with
//                         the state gradient in shared memory, starting from
//                         the sum of its children's initial-state gradients.
//   gdn_bwd_chunk_kernel  one CTA per (chunk, head): everything above that
//                         needs only the chunk and its two state (gradient)s.
//   gdn_bwd_token_kernel  one block per (64 tokens, q / k / v head): the
//                         convolution's input gradient (scattered to the
//                         path's previous tokens) and weight gradient.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "gdn_common.h"
#include "internal.h"
#include "layout.h"

namespace stp {
namespace {

constexpr int kD = kGdnD, kC = kGdnChunk;
constexpr int kBT = 256;   // threads of every backward kernel

struct GbParams {
  int N, H, C, seg0;
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
  const float* s0;           // [rows, d, d]
  float* dsend;              // [rows, d, d]
  float* dvp;                // [rows, 64, d]
  float* sgrad;              // [n_seg H, d, d]
  float* dqkv;               // [N, C]
  float* scr;                // [rows, 2, 64, d]  V', dW
  float* dx;                 // [N, C]
  float* dconv_w;            // [C, 4]
  float* dg;                 // [N, H]
  float* dbeta;              // [N, H]
};

__device__ __forceinline__ float bf(const __nv_bfloat16* p) { return __bfloat162float(*p); }

// C (M x N) = sum_{k < K} A(m, k) B(k, n) by 256 threads on a 16 x 16 grid;
// each thread holds rows tm + 16 i and columns tn + 16 j and hands every
// result to store(m, n, value).  The (m, n) -> thread map depends on M and
// N only, so passes of the same shape may read-modify-write their outputs.
template <int M, int N, typename FA, typename FB, typename FS>
__device__ __forceinline__ void bgemm(int K, FA A, FB B, FS store) {
  constexpr int RM = M / 16, RN = N / 16;
  const int tm = threadIdx.x >> 4, tn = threadIdx.x & 15;
  float acc[RM][RN];
#pragma unroll
  for (int i = 0; i < RM; ++i)
#pragma unroll
    for (int j = 0; j < RN; ++j) acc[i][j] = 0.f;
#pragma unroll 8   // loads of eight k steps in flight: the operands mostly come from L2
  for (int k = 0; k < K; ++k) {
    float a[RM], b[RN];
#pragma unroll
    for (int i = 0; i < RM; ++i) a[i] = A(tm + 16 * i, k);
#pragma unroll
    for (int j = 0; j < RN; ++j) b[j] = B(k, tn + 16 * j);
#pragma unroll
    for (int i = 0; i < RM; ++i)
#pragma unroll
      for (int j = 0; j < RN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
  }
#pragma unroll
  for (int i = 0; i < RM; ++i)
#pragma unroll
    for (int j = 0; j < RN; ++j) store(tm + 16 * i, tn + 16 * j, acc[i][j]);
}

// ---------------------------------------------------------------------------
// Reverse walk of one (segment, head).
constexpr int kWalkSmem = (2 * kD * kD + kC * kD) * 4 + (3 * kC * kD + kC * kC) * 2;

__global__ void __launch_bounds__(kBT, 1) gdn_bwd_walk_kernel(const GbParams p) {
  extern __shared__ float wsm[];
  float* dS = wsm;                       // [128][128]
  float* dSn = dS + kD * kD;             // [128][128]
  float* sdVp = dSn + kD * kD;           // [64][128]
  __nv_bfloat16* sQt = reinterpret_cast<__nv_bfloat16*>(sdVp + kC * kD);   // [64][128]
  __nv_bfloat16* sW = sQt + kC * kD;     // [64][128]
  __nv_bfloat16* sKt = sW + kC * kD;     // [64][128]
  __nv_bfloat16* sP = sKt + kC * kD;     // [64][64]
  const int tid = threadIdx.x;
  const int seg = p.seg0 + (int)(blockIdx.x / p.H), h = (int)(blockIdx.x % p.H);
  const int c0 = p.seg_chunk0[seg], nck = (p.seg_len[seg] + kC - 1) / kC;

  // the segment's end: the sum of its children's initial-state gradients
  const int k0 = p.child_off[seg], k1 = p.child_off[seg + 1];
  for (int e = tid; e < kD * kD; e += kBT) {
    float a = 0.f;
    for (int c = k0; c < k1; ++c) a += p.sgrad[((size_t)p.child[c] * p.H + h) * kD * kD + e];
    dS[e] = a;
  }
  for (int i = nck - 1; i >= 0; --i) {
    const int c = c0 + i, L = p.chunk_len[c], x0 = p.chunk_start[c];
    const size_t row = (size_t)c * p.H + h;
    const float dec = p.decay[row];
    const uint4* wq4 = reinterpret_cast<const uint4*>(p.wq + row * 128 * kD);
    const uint4* kt4 = reinterpret_cast<const uint4*>(p.kt + row * kC * kD);
    const uint4* pm4 = reinterpret_cast<const uint4*>(p.pm + row * kC * kC);
    for (int e = tid; e < kC * kD / 8; e += kBT) {
      reinterpret_cast<uint4*>(sQt)[e] = wq4[e];
      reinterpret_cast<uint4*>(sW)[e] = wq4[kC * kD / 8 + e];
      reinterpret_cast<uint4*>(sKt)[e] = kt4[e];
    }
    for (int e = tid; e < kC * kC / 8; e += kBT) reinterpret_cast<uint4*>(sP)[e] = pm4[e];
    __syncthreads();   // dS complete (children's sum or the previous chunk's dS0)
    float4* de = reinterpret_cast<float4*>(p.dsend + row * kD * kD);
    for (int e = tid; e < kD * kD / 4; e += kBT) de[e] = reinterpret_cast<const float4*>(dS)[e];
    const float* dO = p.d_o + ((size_t)x0 * p.H + h) * kD;
    const size_t dOs = (size_t)p.H * kD;   // token stride of dO
    // dV' = P^T dO + K~ dS   (rows t >= L: P and K~ rows are zero)
    float* gdvp = p.dvp + row * kC * kD;
    bgemm<kC, kD>(
        kC + kD,
        [&](int m, int k) { return k < kC ? bf(sP + k * kC + m) : bf(sKt + m * kD + (k - kC)); },
        [&](int k, int n) { return k < kC ? (k < L ? dO[k * dOs + n] : 0.f) : dS[(k - kC) * kD + n]; },
        [&](int m, int n, float v) {
          sdVp[m * kD + n] = v;
          gdvp[m * kD + n] = v;
        });
    __syncthreads();
    // dS0 = Q~^T dO + e^{gam_n} dS - W^T dV'
    bgemm<kD, kD>(
        2 * kC,
        [&](int m, int k) { return k < kC ? bf(sQt + k * kD + m) : -bf(sW + (k - kC) * kD + m); },
        [&](int k, int n) { return k < kC ? (k < L ? dO[k * dOs + n] : 0.f) : sdVp[(k - kC) * kD + n]; },
        [&](int m, int n, float v) { dSn[m * kD + n] = v + dec * dS[m * kD + n]; });
    __syncthreads();
    float* t = dS;
    dS = dSn;
    dSn = t;
  }
  float4* sg = reinterpret_cast<float4*>(p.sgrad + ((size_t)seg * p.H + h) * kD * kD);
  for (int e = tid; e < kD * kD / 4; e += kBT) sg[e] = reinterpret_cast<const float4*>(dS)[e];
}

// ---------------------------------------------------------------------------
// Chunk-local gradients of one (chunk, head).
constexpr int kChunkSmem = 8 * kC * kC * 4 + 6 * kC * 4;

__global__ void __launch_bounds__(kBT, 1) gdn_bwd_chunk_kernel(const GbParams p) {
  extern __shared__ float csm[];
  float* sKK = csm;                 // each [64][64]
  float* sQK = sKK + kC * kC;
  float* sA = sQK + kC * kC;
  float* sT = sA + kC * kC;
  float* sdP = sT + kC * kC;
  float* sdT = sdP + kC * kC;
  float* sX = sdT + kC * kC;
  float* sdA = sX + kC * kC;
  float* gam = sdA + kC * kC;       // each [64]
  float* bt = gam + kC;
  float* eg = bt + kC;
  float* ek = eg + kC;
  float* dgam = ek + kC;
  float* dbt = dgam + kC;
  const int tid = threadIdx.x;
  const int ch = (int)(blockIdx.x / p.H), h = (int)(blockIdx.x % p.H);
  const int x0 = p.chunk_start[ch], L = p.chunk_len[ch];
  const size_t row = (size_t)ch * p.H + h;
  const int Hd = p.H * kD;
  const float sc = p.scale;
  const __nv_bfloat16* yq = p.y + (size_t)x0 * p.C + h * kD;
  auto q = [&](int t, int k) { return t < L ? bf(yq + (size_t)t * p.C + k) : 0.f; };
  auto kk = [&](int t, int k) { return t < L ? bf(yq + (size_t)t * p.C + Hd + k) : 0.f; };
  auto vv = [&](int t, int k) { return t < L ? bf(yq + (size_t)t * p.C + 2 * Hd + k) : 0.f; };
  const float* S0 = p.s0 + row * kD * kD;
  const float* dSe = p.dsend + row * kD * kD;
  const float* dVp = p.dvp + row * kC * kD;
  const float* dOb = p.d_o + ((size_t)x0 * p.H + h) * kD;
  const size_t dOs = (size_t)p.H * kD;
  auto dO = [&](int t, int j) { return t < L ? dOb[t * dOs + j] : 0.f; };
  const float* Uh = p.ut + row * kD * kC;   // U^[t][j] at j * 64 + t
  const __nv_bfloat16* Wb = p.wq + (row * 128 + kC) * kD;
  float* Vp = p.scr + row * 2 * kC * kD;
  float* dW = Vp + kC * kD;
  float* dq = p.dqkv + (size_t)x0 * p.C + h * kD;
  float* dk = dq + Hd;
  float* dv = dq + 2 * Hd;

  if (tid < 32) {   // gam = inclusive prefix sum of g; beta; e^gam; e^{gam_n - gam}
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
  }
  if (tid < kC) {
    bt[tid] = tid < L ? p.beta[(size_t)(x0 + tid) * p.H + h] : 0.f;
    dgam[tid] = 0.f;
    dbt[tid] = 0.f;
  }
  __syncthreads();
  // K K^T, Q K^T
  bgemm<kC, kC>(kD, [&](int m, int k) { return kk(m, k); }, [&](int k, int n) { return kk(n, k); },
                [&](int m, int n, float v) { sKK[m * kC + n] = v; });
  bgemm<kC, kC>(kD, [&](int m, int k) { return q(m, k); }, [&](int k, int n) { return kk(n, k); },
                [&](int m, int n, float v) { sQK[m * kC + n] = v; });
  __syncthreads();
  for (int e = tid; e < kC * kC; e += kBT) {
    const int t = e / kC, s = e % kC;
    sA[e] = (s < t && t < L) ? bt[t] * expf(gam[t] - gam[s]) * sKK[e] : 0.f;
  }
  __syncthreads();
  if (tid < kC) {   // T = (I + A)^{-1}, column tid, by forward substitution
    const int j = tid;
    for (int t = 0; t < kC; ++t) {
      float x = t == j ? 1.f : 0.f;
      for (int s = j; s < t; ++s) x = fmaf(-sA[t * kC + s], sT[s * kC + j], x);
      sT[t * kC + j] = x;
    }
  }
  __syncthreads();
  // V' = U^ - W S0
  bgemm<kC, kD>(kD, [&](int m, int k) { return bf(Wb + m * kD + k); }, [&](int k, int n) { return S0[k * kD + n]; },
                [&](int m, int n, float v) { Vp[m * kD + n] = Uh[n * kC + m] - v; });
  __syncthreads();
  // dP = dO V'^T;  dW = -dV' S0^T
  bgemm<kC, kC>(kD, [&](int m, int k) { return dO(m, k); }, [&](int k, int n) { return Vp[n * kD + k]; },
                [&](int m, int n, float v) { sdP[m * kC + n] = v; });
  bgemm<kC, kD>(kD, [&](int m, int k) { return dVp[m * kD + k]; }, [&](int k, int n) { return S0[n * kD + k]; },
                [&](int m, int n, float v) { dW[m * kD + n] = -v; });
  __syncthreads();
  // dT = dV' (beta V)^T + dW (beta e^gam K)^T
  bgemm<kC, kC>(
      2 * kD, [&](int m, int k) { return k < kD ? dVp[m * kD + k] : dW[m * kD + (k - kD)]; },
      [&](int k, int n) { return k < kD ? bt[n] * vv(n, k) : bt[n] * eg[n] * kk(n, k - kD); },
      [&](int m, int n, float v) { sdT[m * kC + n] = v; });
  __syncthreads();
  bgemm<kC, kC>(kC, [&](int m, int k) { return sT[k * kC + m]; }, [&](int k, int n) { return sdT[k * kC + n]; },
                [&](int m, int n, float v) { sX[m * kC + n] = v; });
  __syncthreads();
  bgemm<kC, kC>(kC, [&](int m, int k) { return sX[m * kC + k]; }, [&](int k, int n) { return sT[n * kC + k]; },
                [&](int m, int n, float v) { sdA[m * kC + n] = (n < m && m < L) ? -v : 0.f; });
  __syncthreads();

  // dq = scale e^gam dQ~ + scale (dP o Gamma) K, with dgam += dQ~ . Q~
  bgemm<kC, kD>(kD, [&](int m, int k) { return dO(m, k); }, [&](int k, int n) { return S0[n * kD + k]; },
                [&](int m, int n, float v) {
                  if (m < L) {
                    dq[(size_t)m * p.C + n] = sc * eg[m] * v;
                    atomicAdd(&dgam[m], v * sc * eg[m] * q(m, n));
                  }
                });
  bgemm<kC, kD>(
      kC, [&](int m, int k) { return k <= m ? sc * sdP[m * kC + k] * expf(gam[m] - gam[k]) : 0.f; },
      [&](int k, int n) { return kk(k, n); },
      [&](int m, int n, float v) {
        if (m < L) dq[(size_t)m * p.C + n] += v;
      });
  // dk = e^{gam_n - gam} dK~ (dK~ = V' dS_n^T), with the K~ terms of dgam
  bgemm<kC, kD>(kD, [&](int m, int k) { return Vp[m * kD + k]; }, [&](int k, int n) { return dSe[n * kD + k]; },
                [&](int m, int n, float v) {
                  if (m < L) {
                    dk[(size_t)m * p.C + n] = ek[m] * v;
                    const float c = v * ek[m] * kk(m, n);
                    atomicAdd(&dgam[m], -c);
                    atomicAdd(&dgam[L - 1], c);
                  }
                });
  // + scale (dP o Gamma)^T Q
  bgemm<kC, kD>(
      kC, [&](int m, int k) { return m <= k ? sc * sdP[k * kC + m] * expf(gam[k] - gam[m]) : 0.f; },
      [&](int k, int n) { return q(k, n); },
      [&](int m, int n, float v) {
        if (m < L) dk[(size_t)m * p.C + n] += v;
      });
  // + the A terms: M = dA o E (E_ts = e^{gam_t - gam_s}, s < t); dk_t += beta_t M_t. K, dk_s += sum_t beta_t M_ts k_t
  bgemm<kC, kD>(
      kC, [&](int m, int k) { return k < m ? bt[m] * sdA[m * kC + k] * expf(gam[m] - gam[k]) : 0.f; },
      [&](int k, int n) { return kk(k, n); },
      [&](int m, int n, float v) {
        if (m < L) dk[(size_t)m * p.C + n] += v;
      });
  bgemm<kC, kD>(
      kC, [&](int m, int k) { return m < k ? bt[k] * sdA[k * kC + m] * expf(gam[k] - gam[m]) : 0.f; },
      [&](int k, int n) { return kk(k, n); },
      [&](int m, int n, float v) {
        if (m < L) dk[(size_t)m * p.C + n] += v;
      });
  // + beta e^gam dB_W (dB_W = T^T dW), with its beta and gam terms
  bgemm<kC, kD>(kC, [&](int m, int k) { return sT[k * kC + m]; }, [&](int k, int n) { return dW[k * kD + n]; },
                [&](int m, int n, float v) {
                  if (m < L) {
                    const float km = kk(m, n);
                    dk[(size_t)m * p.C + n] += bt[m] * eg[m] * v;
                    atomicAdd(&dbt[m], eg[m] * v * km);
                    atomicAdd(&dgam[m], bt[m] * eg[m] * v * km);
                  }
                });
  // dv = beta dB_U (dB_U = T^T dV'), with its beta term
  bgemm<kC, kD>(kC, [&](int m, int k) { return sT[k * kC + m]; }, [&](int k, int n) { return dVp[k * kD + n]; },
                [&](int m, int n, float v) {
                  if (m < L) {
                    dv[(size_t)m * p.C + n] = bt[m] * v;
                    atomicAdd(&dbt[m], v * vv(m, n));
                  }
                });
  // the P and A terms of dgam, the A term of dbeta
  for (int e = tid; e < kC * kC; e += kBT) {
    const int t = e / kC, s = e % kC;
    if (s <= t && t < L) {
      const float E = expf(gam[t] - gam[s]);
      const float c = sdP[e] * sc * sQK[e] * E;
      atomicAdd(&dgam[t], c);
      atomicAdd(&dgam[s], -c);
      if (s < t) {
        const float c2 = sdA[e] * sA[e];
        atomicAdd(&dgam[t], c2);
        atomicAdd(&dgam[s], -c2);
        atomicAdd(&dbt[t], sdA[e] * E * sKK[e]);
      }
    }
  }
  // the decay term: dgam_{n-1} += e^{gam_n} <dS_n, S0>
  {
    float part = 0.f;
    for (int e = tid; e < kD * kD; e += kBT) part = fmaf(dSe[e], S0[e], part);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    if ((tid & 31) == 0) atomicAdd(&dgam[L - 1], eg[L - 1] * part);
  }
  __syncthreads();
  if (tid < 32) {   // dg = reverse cumulative sum of dgam over the chunk's tokens
    float a = tid + 32 < L ? dgam[tid + 32] : 0.f, b = tid < L ? dgam[tid] : 0.f;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float ua = __shfl_down_sync(0xffffffffu, a, off), ub = __shfl_down_sync(0xffffffffu, b, off);
      if (tid + off < 32) {
        a += ua;
        b += ub;
      }
    }
    b += __shfl_sync(0xffffffffu, a, 0);   // the whole upper half
    if (tid < L) {
      p.dg[(size_t)(x0 + tid) * p.H + h] = b;
      p.dbeta[(size_t)(x0 + tid) * p.H + h] = dbt[tid];
    }
    if (tid + 32 < L) {
      p.dg[(size_t)(x0 + tid + 32) * p.H + h] = a;
      p.dbeta[(size_t)(x0 + tid + 32) * p.H + h] = dbt[tid + 32];
    }
  }
}

// ---------------------------------------------------------------------------
// Back through the unit-norm heads, SiLU and the path convolution.
__global__ void __launch_bounds__(kBT) gdn_bwd_token_kernel(const GbParams p) {
  __shared__ float red[16][16][33];   // [token lane][vector][8 channels x 4 taps]
  const int grp = blockIdx.y, lt = threadIdx.x >> 4, vec = threadIdx.x & 15;
  const int ch = grp * kD + vec * 8;
  const bool is_qk = grp < 2 * p.H;
  float4 wv[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) wv[i] = reinterpret_cast<const float4*>(p.conv_w)[ch + i];
  float dw[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int t = 0; t < 4; ++t) dw[i][t] = 0.f;
  const unsigned grpmask = 0xffffu << (threadIdx.x & 16);
#pragma unroll 1
  for (int it = 0; it < 4; ++it) {
    const int x = blockIdx.x * 64 + it * 16 + lt;
    const int p1 = x < p.N ? p.prev[x] : -2;
    if (p1 == -2) continue;   // a pad or past the end: the same for all 16 lanes of the token
    const int src[4] = {p.prev3[x], p.prev2[x], p1, x};
    float z[8], xin[4][8];
#pragma unroll
    for (int i = 0; i < 8; ++i) z[i] = 0.f;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
#pragma unroll
      for (int i = 0; i < 8; ++i) xin[t][i] = 0.f;
      if (src[t] < 0) continue;
      const __nv_bfloat16* xr = p.x + (size_t)src[t] * p.C + ch;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        xin[t][i] = __bfloat162float(xr[i]);
        const float w = t == 0 ? wv[i].x : t == 1 ? wv[i].y : t == 2 ? wv[i].z : wv[i].w;
        z[i] = fmaf(w, xin[t][i], z[i]);
      }
    }
    float sg[8], y[8], dy[8];
    const float* dyin = p.dqkv + (size_t)x * p.C + ch;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      sg[i] = 1.f / (1.f + expf(-z[i]));
      y[i] = z[i] * sg[i];
      dy[i] = dyin[i];
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
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float dz = dy[i] * sg[i] * (1.f + z[i] * (1.f - sg[i]));
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        if (src[t] < 0) continue;
        const float w = t == 0 ? wv[i].x : t == 1 ? wv[i].y : t == 2 ? wv[i].z : wv[i].w;
        atomicAdd(p.dx + (size_t)src[t] * p.C + ch + i, w * dz);
        dw[i][t] = fmaf(xin[t][i], dz, dw[i][t]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int t = 0; t < 4; ++t) red[lt][vec][i * 4 + t] = dw[i][t];
  __syncthreads();
  if (threadIdx.x < 16 * 32) {
    for (int e = threadIdx.x; e < 16 * 32; e += kBT) {
      const int vv = e / 32, j = e % 32;
      float a = 0.f;
      for (int l = 0; l < 16; ++l) a += red[l][vv][j];
      atomicAdd(p.dconv_w + (size_t)(grp * kD + vv * 8 + j / 4) * 4 + (j % 4), a);
    }
  }
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
  if (e == cudaSuccess && N > 0) e = cudaMemsetAsync(dx, 0, (size_t)N * C * 4, s);
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
  p.scr = reinterpret_cast<float*>(ws + Lw.scr);
  p.dx = dx;
  p.dconv_w = dconv_w;
  p.dg = dg;
  p.dbeta = dbeta;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(gdn_bwd_walk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kWalkSmem);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(gdn_bwd_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kChunkSmem);
  });
  if (attr_err != cudaSuccess) return fail(STP_ECUDA, "stp_gdn_bwd: %s", cudaGetErrorString(attr_err));
  // pads keep dq^, dk^, dv = 0 (the chunk kernel writes real tokens only)
  e = cudaMemsetAsync(p.dqkv, 0, (size_t)N * C * 4, s);
  if (e != cudaSuccess) return fail(STP_ECUDA, "stp_gdn_bwd: %s", cudaGetErrorString(e));
  const int32_t* depth_off = w + w[GP_DEPTH_OFF];
  for (int d = n_depth - 1; d >= 0; --d) {
    const int n = depth_off[d + 1] - depth_off[d];
    if (n <= 0) continue;
    p.seg0 = depth_off[d];
    gdn_bwd_walk_kernel<<<(unsigned)(n * H), kBT, kWalkSmem, s>>>(p);
  }
  if (n_chunk > 0) gdn_bwd_chunk_kernel<<<(unsigned)(n_chunk * H), kBT, kChunkSmem, s>>>(p);
  gdn_bwd_token_kernel<<<dim3((unsigned)((N + 63) / 64), (unsigned)(3 * H)), kBT, 0, s>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(STP_ECUDA, "stp_gdn_bwd: %s", cudaGetErrorString(e));
  return STP_OK;
}
