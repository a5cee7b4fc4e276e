// Tree attention on CUDA cores (FFMA), driven by the tile lists of
// stp_classify.  This is the float32 path (head_dim 64 or 128).
//
// Forward: one block per (query tile, query head, row); two threads per
// query, each holding half of the head dimension (the dot product is joined
// with one shuffle).  Key/value tiles of the query tile's list are staged in
// shared memory; keys are consumed 32 at a time with an online softmax in
// base 2 (scores pre-multiplied by scale * log2 e).  The visibility
// predicate j <= i && se[j] >= i is evaluated on PARTIAL tiles only.
//
// Backward: Delta = rowsum(dO * O); dK/dV with one block per (key tile, kv
// head, row) walking the key tile's list of query tiles for every query head
// of the group; dQ with one block per (query tile, query head, row) walking
// the query tile's list of key tiles.  No atomics: every output element is
// written by exactly one thread.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "layout.h"
#include "simt.h"

namespace stp {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Loads rows [row0, row0+n) of one head of a [R, T, H, D] tensor into
// shared memory with row stride `ld` floats.
template <typename Tin, int D>
__device__ __forceinline__ void stage_rows(float* dst, int ld, const Tin* src, size_t row_base,
                                           int H, int head, int n, int tid, int nthreads) {
  for (int idx = tid; idx < n * D; idx += nthreads) {
    const int rr = idx / D, c = idx - rr * D;
    dst[rr * ld + c] = to_f(src[((row_base + rr) * H + head) * D + c]);
  }
}

template <typename Tin, int D>
__global__ void __launch_bounds__(256) fwd_simt_kernel(AttnArgs a) {
  constexpr int DH = D / 2;
  extern __shared__ float sm[];
  float* Ks = sm;                  // [128][D]
  float* Vs = Ks + kTile * D;      // [128][D]
  int* se_s = reinterpret_cast<int*>(Vs + kTile * D);
  const int qt = blockIdx.x, h = blockIdx.y, r = blockIdx.z;
  const int tid = threadIdx.x, t = tid >> 1, half = tid & 1;
  const int T = a.T, NT = T / kTile, G = a.Hq / a.Hkv, g = h / G;
  const int i = qt * kTile + t;
  const size_t rowT = (size_t)r * T;
  const Tin* Q = static_cast<const Tin*>(a.q);
  const Tin* K = static_cast<const Tin*>(a.k);
  const Tin* V = static_cast<const Tin*>(a.v);
  const float qs = a.scale * kLog2e;
  float qv[DH], o[DH];
#pragma unroll
  for (int d = 0; d < DH; ++d) {
    qv[d] = to_f(Q[((rowT + i) * a.Hq + h) * D + half * DH + d]) * qs;
    o[d] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  const int cnt = a.csr_cnt[(size_t)r * NT + qt];
  const int32_t* list = a.csr + ((size_t)r * NT + qt) * NT;
  for (int e = 0; e < cnt; ++e) {
    const int ent = list[e], kt = ent >> 1, part = ent & 1, k0 = kt * kTile;
    if (kt < 0 || kt >= NT) {
      if (tid == 0) atomicOr(a.err, kErrBadList);
      break;
    }
    __syncthreads();
    stage_rows<Tin, D>(Ks, D, K, rowT + k0, a.Hkv, g, kTile, tid, 256);
    stage_rows<Tin, D>(Vs, D, V, rowT + k0, a.Hkv, g, kTile, tid, 256);
    if (tid < kTile) se_s[tid] = a.se[rowT + k0 + tid];
    __syncthreads();
    for (int c0 = 0; c0 < kTile; c0 += 32) {
      float s[32];
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float* kr = Ks + (c0 + c) * D + half * DH;
        float acc = 0.f;
#pragma unroll
        for (int d = 0; d < DH; ++d) acc = fmaf(qv[d], kr[d], acc);
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        const int j = k0 + c0 + c;
        const bool vis = !part || (j <= i && se_s[c0 + c] >= i);
        s[c] = vis ? acc : -INFINITY;
        mx = fmaxf(mx, s[c]);
      }
      const float mn = fmaxf(m, mx);
      if (mn == -INFINITY) continue;
      const float alpha = exp2f(m - mn);
      l *= alpha;
#pragma unroll
      for (int d = 0; d < DH; ++d) o[d] *= alpha;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float p = exp2f(s[c] - mn);
        l += p;
        const float* vr = Vs + (c0 + c) * D + half * DH;
#pragma unroll
        for (int d = 0; d < DH; ++d) o[d] = fmaf(p, vr[d], o[d]);
      }
      m = mn;
    }
  }
  Tin* O = static_cast<Tin*>(a.o);
  const float inv = 1.f / l;
#pragma unroll
  for (int d = 0; d < DH; ++d) O[((rowT + i) * a.Hq + h) * D + half * DH + d] = from_f<Tin>(o[d] * inv);
  if (half == 0) a.lse[((size_t)r * a.Hq + h) * T + i] = (m + log2f(l)) * kLn2;
}

// Delta[r,h,i] = sum_d dO * O; one warp per (r, i, h) row.
template <typename Tin, int D>
__global__ void __launch_bounds__(256) delta_kernel(AttnArgs a) {
  const int lane = threadIdx.x & 31;
  const size_t rows = (size_t)a.R * a.T * a.Hq;
  const Tin* O = static_cast<const Tin*>(a.o_in);
  const Tin* dO = static_cast<const Tin*>(a.dout);
  for (size_t w = (size_t)blockIdx.x * 8 + (threadIdx.x >> 5); w < rows; w += (size_t)gridDim.x * 8) {
    float acc = 0.f;
    for (int d = lane; d < D; d += 32) acc = fmaf(to_f(O[w * D + d]), to_f(dO[w * D + d]), acc);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) {
      const int h = (int)(w % a.Hq);
      const size_t ri = w / a.Hq;  // r * T + i
      const size_t r = ri / a.T, i = ri - r * a.T;
      a.delta[(r * a.Hq + h) * a.T + i] = acc;
    }
  }
}

constexpr int kChunk = 32;  // query / key rows staged per step in the backward

template <typename Tin, int D>
__global__ void __launch_bounds__(256) dkdv_simt_kernel(AttnArgs a) {
  constexpr int DH = D / 2, LD = D + 1;
  extern __shared__ float sm[];
  float* Kown = sm;                 // [128][D+1]
  float* Vown = Kown + kTile * LD;  // [128][D+1]
  float* Qc = Vown + kTile * LD;    // [32][D]
  float* dOc = Qc + kChunk * D;     // [32][D]
  float* lse2 = dOc + kChunk * D;   // [32]
  float* dlt = lse2 + kChunk;       // [32]
  const int kt = blockIdx.x, g = blockIdx.y, r = blockIdx.z;
  const int tid = threadIdx.x, t = tid >> 1, half = tid & 1;
  const int T = a.T, NT = T / kTile, G = a.Hq / a.Hkv;
  const int j = kt * kTile + t;
  const size_t rowT = (size_t)r * T;
  const Tin* Q = static_cast<const Tin*>(a.q);
  const Tin* K = static_cast<const Tin*>(a.k);
  const Tin* V = static_cast<const Tin*>(a.v);
  const Tin* dO = static_cast<const Tin*>(a.dout);
  stage_rows<Tin, D>(Kown, LD, K, rowT + kt * kTile, a.Hkv, g, kTile, tid, 256);
  stage_rows<Tin, D>(Vown, LD, V, rowT + kt * kTile, a.Hkv, g, kTile, tid, 256);
  const int sej = a.se[rowT + j];
  const float qs = a.scale * kLog2e;
  float dk[DH], dv[DH];
#pragma unroll
  for (int d = 0; d < DH; ++d) dk[d] = dv[d] = 0.f;
  const int cnt = a.csc_cnt[(size_t)r * NT + kt];
  const int32_t* list = a.csc + ((size_t)r * NT + kt) * NT;
  const float* kr = Kown + t * LD + half * DH;
  const float* vr = Vown + t * LD + half * DH;
  for (int e = 0; e < cnt; ++e) {
    const int ent = list[e], qt = ent >> 1, part = ent & 1;
    if (qt < 0 || qt >= NT) {
      if (tid == 0) atomicOr(a.err, kErrBadList);
      break;
    }
    for (int hh = 0; hh < G; ++hh) {
      const int h = g * G + hh;
      for (int c0 = 0; c0 < kTile; c0 += kChunk) {
        const int i0 = qt * kTile + c0;
        __syncthreads();
        stage_rows<Tin, D>(Qc, D, Q, rowT + i0, a.Hq, h, kChunk, tid, 256);
        stage_rows<Tin, D>(dOc, D, dO, rowT + i0, a.Hq, h, kChunk, tid, 256);
        if (tid < kChunk) {
          lse2[tid] = a.lse[((size_t)r * a.Hq + h) * T + i0 + tid] * kLog2e;
          dlt[tid] = a.delta[((size_t)r * a.Hq + h) * T + i0 + tid];
        }
        __syncthreads();
        for (int c = 0; c < kChunk; ++c) {
          const int i = i0 + c;
          const float* qr = Qc + c * D + half * DH;
          const float* gr = dOc + c * D + half * DH;
          float s = 0.f, dp = 0.f;
#pragma unroll
          for (int d = 0; d < DH; ++d) {
            s = fmaf(qr[d], kr[d], s);
            dp = fmaf(gr[d], vr[d], dp);
          }
          s += __shfl_xor_sync(0xffffffffu, s, 1);
          dp += __shfl_xor_sync(0xffffffffu, dp, 1);
          const bool vis = !part || (j <= i && sej >= i);
          const float p = vis ? exp2f(s * qs - lse2[c]) : 0.f;
          const float ds = p * (dp - dlt[c]);
#pragma unroll
          for (int d = 0; d < DH; ++d) {
            dv[d] = fmaf(p, gr[d], dv[d]);
            dk[d] = fmaf(ds, qr[d], dk[d]);
          }
        }
      }
    }
  }
  Tin* dK = static_cast<Tin*>(a.dk);
  Tin* dV = static_cast<Tin*>(a.dv);
#pragma unroll
  for (int d = 0; d < DH; ++d) {
    dK[((rowT + j) * a.Hkv + g) * D + half * DH + d] = from_f<Tin>(dk[d] * a.scale);
    dV[((rowT + j) * a.Hkv + g) * D + half * DH + d] = from_f<Tin>(dv[d]);
  }
}

template <typename Tin, int D>
__global__ void __launch_bounds__(256) dq_simt_kernel(AttnArgs a) {
  constexpr int DH = D / 2, LD = D + 1;
  extern __shared__ float sm[];
  float* Qown = sm;                   // [128][D+1]
  float* dOown = Qown + kTile * LD;   // [128][D+1]
  float* Kc = dOown + kTile * LD;     // [32][D]
  float* Vc = Kc + kChunk * D;        // [32][D]
  int* sec = reinterpret_cast<int*>(Vc + kChunk * D);
  const int qt = blockIdx.x, h = blockIdx.y, r = blockIdx.z;
  const int tid = threadIdx.x, t = tid >> 1, half = tid & 1;
  const int T = a.T, NT = T / kTile, G = a.Hq / a.Hkv, g = h / G;
  const int i = qt * kTile + t;
  const size_t rowT = (size_t)r * T;
  const Tin* Q = static_cast<const Tin*>(a.q);
  const Tin* K = static_cast<const Tin*>(a.k);
  const Tin* V = static_cast<const Tin*>(a.v);
  const Tin* dO = static_cast<const Tin*>(a.dout);
  stage_rows<Tin, D>(Qown, LD, Q, rowT + qt * kTile, a.Hq, h, kTile, tid, 256);
  stage_rows<Tin, D>(dOown, LD, dO, rowT + qt * kTile, a.Hq, h, kTile, tid, 256);
  const float qs = a.scale * kLog2e;
  const float lse2 = a.lse[((size_t)r * a.Hq + h) * T + i] * kLog2e;
  const float dlt = a.delta[((size_t)r * a.Hq + h) * T + i];
  float dq[DH];
#pragma unroll
  for (int d = 0; d < DH; ++d) dq[d] = 0.f;
  const int cnt = a.csr_cnt[(size_t)r * NT + qt];
  const int32_t* list = a.csr + ((size_t)r * NT + qt) * NT;
  const float* qr = Qown + t * LD + half * DH;
  const float* gr = dOown + t * LD + half * DH;
  for (int e = 0; e < cnt; ++e) {
    const int ent = list[e], kt = ent >> 1, part = ent & 1;
    if (kt < 0 || kt >= NT) {
      if (tid == 0) atomicOr(a.err, kErrBadList);
      break;
    }
    for (int c0 = 0; c0 < kTile; c0 += kChunk) {
      const int j0 = kt * kTile + c0;
      __syncthreads();
      stage_rows<Tin, D>(Kc, D, K, rowT + j0, a.Hkv, g, kChunk, tid, 256);
      stage_rows<Tin, D>(Vc, D, V, rowT + j0, a.Hkv, g, kChunk, tid, 256);
      if (tid < kChunk) sec[tid] = a.se[rowT + j0 + tid];
      __syncthreads();
      for (int c = 0; c < kChunk; ++c) {
        const int j = j0 + c;
        const float* kr = Kc + c * D + half * DH;
        const float* vr = Vc + c * D + half * DH;
        float s = 0.f, dp = 0.f;
#pragma unroll
        for (int d = 0; d < DH; ++d) {
          s = fmaf(qr[d], kr[d], s);
          dp = fmaf(gr[d], vr[d], dp);
        }
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        dp += __shfl_xor_sync(0xffffffffu, dp, 1);
        const bool vis = !part || (j <= i && sec[c] >= i);
        const float p = vis ? exp2f(s * qs - lse2) : 0.f;
        const float ds = p * (dp - dlt);
#pragma unroll
        for (int d = 0; d < DH; ++d) dq[d] = fmaf(ds, kr[d], dq[d]);
      }
    }
  }
  Tin* dQ = static_cast<Tin*>(a.dq);
#pragma unroll
  for (int d = 0; d < DH; ++d) dQ[((rowT + i) * a.Hq + h) * D + half * DH + d] = from_f<Tin>(dq[d] * a.scale);
}

template <typename Tin, int D>
cudaError_t launch_fwd(const AttnArgs& a, cudaStream_t s) {
  const size_t smem = 2 * kTile * D * sizeof(float) + kTile * sizeof(int);
  cudaFuncSetAttribute(fwd_simt_kernel<Tin, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  fwd_simt_kernel<Tin, D><<<dim3(a.T / kTile, a.Hq, a.R), 256, smem, s>>>(a);
  return cudaGetLastError();
}

template <typename Tin, int D>
cudaError_t launch_bwd(const AttnArgs& a, cudaStream_t s) {
  delta_kernel<Tin, D><<<1024, 256, 0, s>>>(a);
  const size_t smem_kv = (2 * kTile * (D + 1) + 2 * kChunk * D + 2 * kChunk) * sizeof(float);
  cudaFuncSetAttribute(dkdv_simt_kernel<Tin, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_kv);
  dkdv_simt_kernel<Tin, D><<<dim3(a.T / kTile, a.Hkv, a.R), 256, smem_kv, s>>>(a);
  const size_t smem_q = (2 * kTile * (D + 1) + 2 * kChunk * D) * sizeof(float) + kChunk * sizeof(int);
  cudaFuncSetAttribute(dq_simt_kernel<Tin, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_q);
  dq_simt_kernel<Tin, D><<<dim3(a.T / kTile, a.Hq, a.R), 256, smem_q, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t simt_fwd(const AttnArgs& a, bool bf16, cudaStream_t s) {
  if (bf16) return a.D == 64 ? launch_fwd<__nv_bfloat16, 64>(a, s) : launch_fwd<__nv_bfloat16, 128>(a, s);
  return a.D == 64 ? launch_fwd<float, 64>(a, s) : launch_fwd<float, 128>(a, s);
}

cudaError_t simt_bwd(const AttnArgs& a, bool bf16, cudaStream_t s) {
  if (bf16) return a.D == 64 ? launch_bwd<__nv_bfloat16, 64>(a, s) : launch_bwd<__nv_bfloat16, 128>(a, s);
  return a.D == 64 ? launch_bwd<float, 64>(a, s) : launch_bwd<float, 128>(a, s);
}

}  // namespace stp
