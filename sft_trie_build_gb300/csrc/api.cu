// C ABI of the tree-attention calls: argument checks, workspace carving and
// dispatch to the kernels.  float32 runs on the CUDA-core kernels; bf16 with
// head_dim 128 runs on the tcgen05 tensor-core kernels.
#include <cuda_runtime.h>

#include "internal.h"
#include "layout.h"
#include "simt.h"
#include "tc.h"

namespace stp {

stp_status check_desc(const stp_attn_desc* d) {
  if (!d) return fail(STP_EINVAL, "attention descriptor is NULL");
  if (d->n_rows < 0) return fail(STP_EINVAL, "n_rows < 0");
  if (d->row_len <= 0 || d->row_len % kTile || d->row_len > kMaxRowLen)
    return fail(STP_EUNSUPPORTED, "row_len %d must be a positive multiple of 128 and <= %d",
                d->row_len, kMaxRowLen);
  if ((d->block_m && d->block_m != kTile) || (d->block_n && d->block_n != kTile))
    return fail(STP_EUNSUPPORTED, "block_m / block_n must be 128");
  if (d->n_q_heads <= 0 || d->n_kv_heads <= 0 || d->n_q_heads % d->n_kv_heads)
    return fail(STP_EUNSUPPORTED, "need n_q_heads %% n_kv_heads == 0 (got %d, %d)", d->n_q_heads,
                d->n_kv_heads);
  if (d->dtype != STP_BF16 && d->dtype != STP_FP32)
    return fail(STP_EUNSUPPORTED, "dtype %d not supported", d->dtype);
  if (d->dtype == STP_BF16 && d->head_dim != 128)
    return fail(STP_EUNSUPPORTED, "bf16 needs head_dim 128 (got %d)", d->head_dim);
  if (d->dtype == STP_FP32 && d->head_dim != 64 && d->head_dim != 128)
    return fail(STP_EUNSUPPORTED, "fp32 needs head_dim 64 or 128 (got %d)", d->head_dim);
  if (!(d->scale > 0.f) || d->scale > 1e4f) return fail(STP_EINVAL, "scale must be positive");
  if (d->max_tile_pairs < 0) return fail(STP_EINVAL, "max_tile_pairs must be >= 0");
  if (d->ds_groups < 0) return fail(STP_EINVAL, "ds_groups must be >= 0");
  if ((int64_t)d->n_rows * d->row_len * d->n_q_heads * d->head_dim > (int64_t)1 << 40)
    return fail(STP_EUNSUPPORTED, "problem too large");
  return STP_OK;
}

static bool misaligned(const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) & (a - 1); }

static stp_status fill_common(const stp_attn_desc* d, const int32_t* se, const void* tile_meta,
                              AttnArgs& a) {
  a.R = d->n_rows;
  a.T = d->row_len;
  a.Hq = d->n_q_heads;
  a.Hkv = d->n_kv_heads;
  a.D = d->head_dim;
  a.scale = d->scale;
  a.se = se;
  const TileMeta m = tile_meta_layout(d->n_rows, d->row_len / kTile);
  const char* base = static_cast<const char*>(tile_meta);
  a.csr_cnt = reinterpret_cast<const int32_t*>(base + m.csr_cnt);
  a.csr = reinterpret_cast<const int32_t*>(base + m.csr);
  a.csc_cnt = reinterpret_cast<const int32_t*>(base + m.csc_cnt);
  a.csc = reinterpret_cast<const int32_t*>(base + m.csc);
  a.csr_off = reinterpret_cast<const int32_t*>(base + m.csr_off);
  a.row_base = reinterpret_cast<const int32_t*>(base + m.row_base);
  a.csc_pair = reinterpret_cast<const int32_t*>(base + m.csc_pair);
  return STP_OK;
}

}  // namespace stp

using namespace stp;

extern "C" stp_status stp_attn_fwd(const stp_attn_desc* desc, const void* q, const void* k,
                                   const void* v, const int32_t* d_subtree_end,
                                   const void* d_tile_meta, void* o, float* lse, void* d_ws,
                                   void* stream) {
  clear_error();
  stp_status st = check_desc(desc);
  if (st) return st;
  if (!q || !k || !v || !d_subtree_end || !d_tile_meta || !o || !lse || !d_ws)
    return fail(STP_EINVAL, "stp_attn_fwd: NULL device pointer");
  if (misaligned(q, 16) || misaligned(k, 16) || misaligned(v, 16) || misaligned(o, 16) ||
      misaligned(lse, 16) || misaligned(d_tile_meta, 256) || misaligned(d_ws, 256))
    return fail(STP_EINVAL, "stp_attn_fwd: tensors must be 16-byte and workspaces 256-byte aligned");
  if (desc->n_rows == 0) return STP_OK;
  AttnArgs a{};
  fill_common(desc, d_subtree_end, d_tile_meta, a);
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.err = static_cast<uint32_t*>(d_ws);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaMemsetAsync(a.err, 0, 4, s);
  cudaError_t e;
  if (desc->dtype == STP_BF16) {
    e = tc_fwd(a, s);
  } else {
    e = simt_fwd(a, false, s);
  }
  if (e != cudaSuccess) return fail(STP_ECUDA, "stp_attn_fwd: %s", cudaGetErrorString(e));
  return STP_OK;
}

extern "C" stp_status stp_attn_bwd(const stp_attn_desc* desc, const void* q, const void* k,
                                   const void* v, const void* o, const float* lse,
                                   const void* d_o, const int32_t* d_subtree_end,
                                   const void* d_tile_meta, void* dq, void* dk, void* dv,
                                   void* d_ws, void* stream) {
  clear_error();
  stp_status st = check_desc(desc);
  if (st) return st;
  if (!q || !k || !v || !o || !lse || !d_o || !d_subtree_end || !d_tile_meta || !dq || !dk ||
      !dv || !d_ws)
    return fail(STP_EINVAL, "stp_attn_bwd: NULL device pointer");
  if (misaligned(q, 16) || misaligned(k, 16) || misaligned(v, 16) || misaligned(o, 16) ||
      misaligned(lse, 16) || misaligned(d_o, 16) || misaligned(dq, 16) || misaligned(dk, 16) ||
      misaligned(dv, 16) || misaligned(d_tile_meta, 256) || misaligned(d_ws, 256))
    return fail(STP_EINVAL, "stp_attn_bwd: tensors must be 16-byte and workspaces 256-byte aligned");
  if (desc->n_rows == 0) return STP_OK;
  AttnArgs a{};
  fill_common(desc, d_subtree_end, d_tile_meta, a);
  a.q = q;
  a.k = k;
  a.v = v;
  a.o_in = o;
  a.lse = const_cast<float*>(lse);
  a.dout = d_o;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  const int64_t cap = pair_capacity(desc->n_rows, desc->row_len / kTile, desc->max_tile_pairs);
  const BwdWs w = bwd_ws_layout(desc->n_rows, desc->row_len, desc->n_q_heads, desc->n_kv_heads,
                                desc->dtype == STP_BF16, cap, desc->ds_groups);
  char* ws = static_cast<char*>(d_ws);
  a.err = reinterpret_cast<uint32_t*>(ws + w.err);
  a.delta = desc->dtype == STP_BF16 ? nullptr : reinterpret_cast<float*>(ws + w.delta);
  a.sbias = desc->dtype == STP_BF16 ? ws + w.sbias : nullptr;
  a.dbias = desc->dtype == STP_BF16 ? ws + w.dbias : nullptr;
  a.ds = desc->dtype == STP_BF16 ? ws + w.ds : nullptr;
  a.ds_cap = cap;
  a.ds_slots = bwd_groups(desc->n_q_heads, desc->n_kv_heads, desc->ds_groups).slots;
  a.ds_slot_bytes = w.slot_bytes;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaMemsetAsync(a.err, 0, 4, s);
  cudaError_t e;
  if (desc->dtype == STP_BF16) {
    e = tc_bwd(a, s);
  } else {
    e = simt_bwd(a, false, s);
  }
  if (e != cudaSuccess) return fail(STP_ECUDA, "stp_attn_bwd: %s", cudaGetErrorString(e));
  return STP_OK;
}
