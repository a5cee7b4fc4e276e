// One attention training step on host buffers, pipelined over groups of kv
// heads.
//
// Rows and kv-head groups of the packed problem are independent, so the heads
// split into n_chunks groups of whole kv heads, each a smaller problem of the
// same shape with its own contiguous device copies of Q, K, V, dO, O, LSE,
// dQ, dK, dV and its own workspaces.  Three kinds of streams (created once
// per device and kept) run the groups:
//   upload    Q, K, V of group c, then dO of group c-1 (strided 2D copies out
//             of the caller's [R*T, H, D] host rows), so that the first
//             forward can start as soon as its own inputs are in;
//   compute c forward of group c once its Q, K, V are in and the caller's
//             stream has reached the call (subtree_end and tile_meta ready),
//             then its backward once dO is in;
//   download  O and LSE of each group after its forward, dQ, dK, dV after its
//             backward, into the caller's host buffers.
// The copies of one group overlap the kernels of the others; only the first
// group's upload and the last group's gradients stay exposed.  The caller's
// stream waits for everything before the call returns control to it, then a
// one-block kernel ORs every group's device error word into the step's word
// (the first 4 bytes of the scratch, read with stp_device_status).
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"
#include "layout.h"

namespace stp {
namespace {

constexpr int kMaxChunks = 16;
constexpr int kMaxDevices = 64;

struct Pipeline {
  bool ready = false;
  cudaStream_t up = nullptr, dn = nullptr, comp[kMaxChunks] = {};
  cudaEvent_t start = nullptr, in_qkv[kMaxChunks] = {}, in_do[kMaxChunks] = {},
              fwd[kMaxChunks] = {}, bwd[kMaxChunks] = {}, up_done = nullptr, dn_done = nullptr;
};

std::mutex g_mu;
Pipeline g_pipe[kMaxDevices];

cudaError_t make_pipeline(Pipeline& p) {
  if (p.ready) return cudaSuccess;
  const unsigned sf = cudaStreamNonBlocking;
  const unsigned ef = cudaEventDisableTiming;
  cudaError_t e = cudaStreamCreateWithFlags(&p.up, sf);
  if (!e) e = cudaStreamCreateWithFlags(&p.dn, sf);
  for (int c = 0; c < kMaxChunks && !e; ++c) e = cudaStreamCreateWithFlags(&p.comp[c], sf);
  if (!e) e = cudaEventCreateWithFlags(&p.start, ef);
  if (!e) e = cudaEventCreateWithFlags(&p.up_done, ef);
  if (!e) e = cudaEventCreateWithFlags(&p.dn_done, ef);
  for (int c = 0; c < kMaxChunks && !e; ++c) {
    e = cudaEventCreateWithFlags(&p.in_qkv[c], ef);
    if (!e) e = cudaEventCreateWithFlags(&p.in_do[c], ef);
    if (!e) e = cudaEventCreateWithFlags(&p.fwd[c], ef);
    if (!e) e = cudaEventCreateWithFlags(&p.bwd[c], ef);
  }
  p.ready = (e == cudaSuccess);
  return e;
}

// Byte offsets of one group's buffers inside the scratch (all 256-aligned).
struct ChunkLayout {
  size_t q, k, v, d_o, o, lse, dq, dk, dv, fwd_ws, bwd_ws, bwd_err, size;
};

struct StepLayout {
  stp_attn_desc cd;  // the per-group descriptor
  ChunkLayout c;     // offsets relative to the group's base
  size_t head, total;
};

stp_status step_layout(const stp_attn_desc* d, int n_chunks, StepLayout& L) {
  stp_status st = check_desc(d);
  if (st) return st;
  if (n_chunks < 1 || n_chunks > kMaxChunks || d->n_kv_heads % n_chunks)
    return fail(STP_EINVAL, "n_chunks must divide n_kv_heads (%d) and lie in [1, %d] (got %d)",
                d->n_kv_heads, kMaxChunks, n_chunks);
  L.cd = *d;
  L.cd.n_q_heads = d->n_q_heads / n_chunks;
  L.cd.n_kv_heads = d->n_kv_heads / n_chunks;
  size_t tm = 0, fws = 0, bws = 0;
  st = stp_workspace_size(&L.cd, &tm, &fws, &bws);
  if (st) return st;
  const size_t eb = d->dtype == STP_BF16 ? 2 : 4;
  const size_t rows = size_t(d->n_rows) * d->row_len;
  const size_t qb = align256(rows * L.cd.n_q_heads * d->head_dim * eb);
  const size_t kb = align256(rows * L.cd.n_kv_heads * d->head_dim * eb);
  ChunkLayout& c = L.c;
  size_t o = 0;
  c.q = o;      o += qb;
  c.k = o;      o += kb;
  c.v = o;      o += kb;
  c.d_o = o;    o += qb;
  c.o = o;      o += qb;
  c.lse = o;    o += align256(rows * L.cd.n_q_heads * 4);
  c.dq = o;     o += qb;
  c.dk = o;     o += kb;
  c.dv = o;     o += kb;
  c.fwd_ws = o; o += align256(fws);
  c.bwd_ws = o; o += align256(bws);
  c.bwd_err = c.bwd_ws + bwd_ws_layout(d->n_rows, d->row_len, L.cd.n_q_heads, L.cd.n_kv_heads,
                                       d->dtype == STP_BF16,
                                       pair_capacity(d->n_rows, d->row_len / kTile, d->max_tile_pairs),
                                       L.cd.ds_groups)
                             .err;
  c.size = o;
  L.head = 256;
  L.total = L.head + size_t(n_chunks) * c.size;
  return STP_OK;
}

struct ErrWords {
  const uint32_t* w[2 * kMaxChunks];
  int n;
};

__global__ void or_error_words(uint32_t* out, ErrWords words) {
  uint32_t x = 0;
  for (int i = threadIdx.x; i < words.n; i += 32) x |= *words.w[i];
#pragma unroll
  for (int s = 16; s; s >>= 1) x |= __shfl_xor_sync(0xffffffffu, x, s);
  if (threadIdx.x == 0) *out = x;
}

// rows x width bytes between a packed device block and a strided host block
cudaError_t copy_cols(void* dst, size_t dpitch, const void* src, size_t spitch, size_t width,
                      size_t rows, cudaMemcpyKind kind, cudaStream_t s) {
  if (!rows || !width) return cudaSuccess;
  return cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, rows, kind, s);
}

}  // namespace
}  // namespace stp

using namespace stp;

extern "C" stp_status stp_step_scratch_size(const stp_attn_desc* desc, int32_t n_chunks,
                                            size_t* scratch_bytes) {
  clear_error();
  if (!scratch_bytes) return fail(STP_EINVAL, "stp_step_scratch_size: NULL output");
  StepLayout L;
  stp_status st = step_layout(desc, n_chunks, L);
  if (st) return st;
  *scratch_bytes = L.total;
  return STP_OK;
}

extern "C" stp_status stp_attn_step_host(const stp_attn_desc* desc, int32_t n_chunks,
                                         const void* q, const void* k, const void* v,
                                         const void* d_o, const int32_t* d_subtree_end,
                                         const void* d_tile_meta, void* o, float* lse, void* dq,
                                         void* dk, void* dv, void* d_scratch,
                                         size_t scratch_bytes, void* stream) {
  clear_error();
  StepLayout L;
  stp_status st = step_layout(desc, n_chunks, L);
  if (st) return st;
  if (!q || !k || !v || !d_o || !o || !lse || !dq || !dk || !dv || !d_subtree_end ||
      !d_tile_meta || !d_scratch)
    return fail(STP_EINVAL, "stp_attn_step_host: NULL pointer");
  if (reinterpret_cast<uintptr_t>(d_scratch) & 255)
    return fail(STP_EINVAL, "stp_attn_step_host: scratch must be 256-byte aligned");
  if (scratch_bytes < L.total)
    return fail(STP_EINVAL, "stp_attn_step_host: scratch holds %zu bytes, needs %zu", scratch_bytes,
                L.total);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e) return fail(STP_ECUDA, "stp_attn_step_host: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(STP_EUNSUPPORTED, "device %d out of range", dev);

  std::lock_guard<std::mutex> lock(g_mu);
  Pipeline& P = g_pipe[dev];
  e = make_pipeline(P);
  if (e) return fail(STP_ECUDA, "stp_attn_step_host: creating streams: %s", cudaGetErrorString(e));
  cudaStream_t caller = static_cast<cudaStream_t>(stream);
  char* base = static_cast<char*>(d_scratch) + L.head;
  uint32_t* step_err = static_cast<uint32_t*>(d_scratch);

  const stp_attn_desc& cd = L.cd;
  const size_t eb = desc->dtype == STP_BF16 ? 2 : 4;
  const size_t rows = size_t(desc->n_rows) * desc->row_len;
  const size_t D = desc->head_dim;
  const size_t qrow = size_t(desc->n_q_heads) * D * eb, krow = size_t(desc->n_kv_heads) * D * eb;
  const size_t qw = size_t(cd.n_q_heads) * D * eb, kw = size_t(cd.n_kv_heads) * D * eb;
  const size_t T = desc->row_len;
  const size_t lrow = size_t(desc->n_q_heads) * T * 4, lw = size_t(cd.n_q_heads) * T * 4;
  auto at = [&](int c, size_t off) { return base + size_t(c) * L.c.size + off; };
  const char* qh = static_cast<const char*>(q);
  const char* kh = static_cast<const char*>(k);
  const char* vh = static_cast<const char*>(v);
  const char* doh = static_cast<const char*>(d_o);

#define STEP_CUDA(x)                                                                   \
  do {                                                                                 \
    cudaError_t ee = (x);                                                              \
    if (ee) return fail(STP_ECUDA, "stp_attn_step_host: %s", cudaGetErrorString(ee)); \
  } while (0)

  // The upload stream may overwrite a group's buffers only after the previous
  // step's kernels and downloads are done with them; the caller's stream
  // already waited for those (end of the previous call), so ordering the
  // upload after the caller's current position covers it.
  STEP_CUDA(cudaEventRecord(P.start, caller));
  STEP_CUDA(cudaStreamWaitEvent(P.up, P.start, 0));
  auto upload_do = [&](int c) -> cudaError_t {
    cudaError_t r = copy_cols(at(c, L.c.d_o), qw, doh + c * qw, qrow, qw, rows, cudaMemcpyHostToDevice, P.up);
    if (!r) r = cudaEventRecord(P.in_do[c], P.up);
    return r;
  };
  for (int c = 0; c < n_chunks; ++c) {
    STEP_CUDA(copy_cols(at(c, L.c.q), qw, qh + c * qw, qrow, qw, rows, cudaMemcpyHostToDevice, P.up));
    STEP_CUDA(copy_cols(at(c, L.c.k), kw, kh + c * kw, krow, kw, rows, cudaMemcpyHostToDevice, P.up));
    STEP_CUDA(copy_cols(at(c, L.c.v), kw, vh + c * kw, krow, kw, rows, cudaMemcpyHostToDevice, P.up));
    STEP_CUDA(cudaEventRecord(P.in_qkv[c], P.up));
    if (c > 0) STEP_CUDA(upload_do(c - 1));
  }
  STEP_CUDA(upload_do(n_chunks - 1));
  STEP_CUDA(cudaEventRecord(P.up_done, P.up));

  for (int c = 0; c < n_chunks; ++c) {
    cudaStream_t s = P.comp[c];
    STEP_CUDA(cudaStreamWaitEvent(s, P.start, 0));
    STEP_CUDA(cudaStreamWaitEvent(s, P.in_qkv[c], 0));
    st = stp_attn_fwd(&cd, at(c, L.c.q), at(c, L.c.k), at(c, L.c.v), d_subtree_end, d_tile_meta,
                      at(c, L.c.o), reinterpret_cast<float*>(at(c, L.c.lse)), at(c, L.c.fwd_ws), s);
    if (st) return st;
    STEP_CUDA(cudaEventRecord(P.fwd[c], s));
    STEP_CUDA(cudaStreamWaitEvent(s, P.in_do[c], 0));
    st = stp_attn_bwd(&cd, at(c, L.c.q), at(c, L.c.k), at(c, L.c.v), at(c, L.c.o),
                      reinterpret_cast<const float*>(at(c, L.c.lse)), at(c, L.c.d_o), d_subtree_end,
                      d_tile_meta, at(c, L.c.dq), at(c, L.c.dk), at(c, L.c.dv), at(c, L.c.bwd_ws), s);
    if (st) return st;
    STEP_CUDA(cudaEventRecord(P.bwd[c], s));
  }

  STEP_CUDA(cudaStreamWaitEvent(P.dn, P.start, 0));
  char* oh = static_cast<char*>(o);
  char* lh = reinterpret_cast<char*>(lse);
  char* dqh = static_cast<char*>(dq);
  char* dkh = static_cast<char*>(dk);
  char* dvh = static_cast<char*>(dv);
  for (int c = 0; c < n_chunks; ++c) {
    STEP_CUDA(cudaStreamWaitEvent(P.dn, P.fwd[c], 0));
    STEP_CUDA(copy_cols(oh + c * qw, qrow, at(c, L.c.o), qw, qw, rows, cudaMemcpyDeviceToHost, P.dn));
    STEP_CUDA(copy_cols(lh + c * lw, lrow, at(c, L.c.lse), lw, lw, desc->n_rows, cudaMemcpyDeviceToHost, P.dn));
  }
  for (int c = 0; c < n_chunks; ++c) {
    STEP_CUDA(cudaStreamWaitEvent(P.dn, P.bwd[c], 0));
    STEP_CUDA(copy_cols(dqh + c * qw, qrow, at(c, L.c.dq), qw, qw, rows, cudaMemcpyDeviceToHost, P.dn));
    STEP_CUDA(copy_cols(dkh + c * kw, krow, at(c, L.c.dk), kw, kw, rows, cudaMemcpyDeviceToHost, P.dn));
    STEP_CUDA(copy_cols(dvh + c * kw, krow, at(c, L.c.dv), kw, kw, rows, cudaMemcpyDeviceToHost, P.dn));
  }
  STEP_CUDA(cudaEventRecord(P.dn_done, P.dn));

  // the caller's stream continues once every copy is done (the kernels
  // finished before the downloads that follow them)
  STEP_CUDA(cudaStreamWaitEvent(caller, P.up_done, 0));
  STEP_CUDA(cudaStreamWaitEvent(caller, P.dn_done, 0));
  ErrWords w{};
  for (int c = 0; c < n_chunks; ++c) {
    w.w[w.n++] = reinterpret_cast<const uint32_t*>(at(c, L.c.fwd_ws));
    w.w[w.n++] = reinterpret_cast<const uint32_t*>(at(c, L.c.bwd_err));
  }
  or_error_words<<<1, 32, 0, caller>>>(step_err, w);
  STEP_CUDA(cudaGetLastError());
#undef STEP_CUDA
  return STP_OK;
}
