// Pieces shared by the Gated DeltaNet forward (gdn.cu) and backward
// (gdn_bwd.cu): descriptor and plan checks, and the device workspace layout.
#pragma once

#include <cmath>
#include <cstdint>

#include "internal.h"
#include "layout.h"

namespace stp {

constexpr int kGdnD = 128;   // head dim

// Workspace (256-byte aligned regions; the error word at offset 0).  The
// forward uses y .. state; a training forward also keeps every chunk's
// starting state (s0) for the backward, which adds its own buffers.
struct GdnLayout {
  size_t y, wq, kt, pm, ut, decay, state, total;          // forward
  size_t s0, dsend, dvp, sgrad, dqkv, dwp, train_total;   // training
};

inline GdnLayout gdn_layout(int64_t N, int H, int64_t n_chunk, int64_t n_seg) {
  GdnLayout L;
  size_t o = 256;
  const int64_t C = 3LL * H * kGdnD, rows = n_chunk * H;
  auto take = [&](size_t& at, size_t bytes) {
    at = o;
    o += align256(bytes);
  };
  take(L.y, (size_t)N * C * 2);                       // conv output q^ | k^ | v, bf16
  take(L.wq, (size_t)rows * 128 * kGdnD * 2);         // [Q~; W] per (chunk, head), bf16
  take(L.kt, (size_t)rows * kGdnChunk * kGdnD * 2);   // K~
  take(L.pm, (size_t)rows * kGdnChunk * kGdnChunk * 2);   // P
  take(L.ut, (size_t)rows * kGdnD * kGdnChunk * 4);   // U^ transposed, float32
  take(L.decay, (size_t)rows * 4);                    // e^{gam_L}
  take(L.state, (size_t)n_seg * H * kGdnD * kGdnD * 4);   // final state of each (segment, head)
  L.total = o;
  take(L.s0, (size_t)rows * kGdnD * kGdnD * 4);       // starting state of each (chunk, head), [d_v][d_k]
  take(L.dsend, (size_t)rows * kGdnD * kGdnD * 4);    // state gradient at each chunk's end, [d_v][d_k]
  take(L.dvp, (size_t)rows * kGdnChunk * kGdnD * 4);  // dV' per (chunk, head), [d_v][64]
  take(L.sgrad, (size_t)n_seg * H * kGdnD * kGdnD * 4);   // state gradient at each segment's start, [d_v][d_k]
  take(L.dqkv, (size_t)N * C * 4);                    // dq^ | dk^ | dv, then dz (the convolution's output gradient)
  take(L.dwp, (size_t)((N + 63) / 64) * C * 4 * 4);   // convolution weight gradient per 64-token block
  L.train_total = o;
  return L;
}

inline stp_status check_gdn_desc(const stp_gdn_desc* d) {
  if (!d) return fail(STP_EINVAL, "GDN descriptor is NULL");
  if (d->n_rows < 0 || d->row_len <= 0 || (int64_t)d->n_rows * d->row_len > (1 << 26))
    return fail(STP_EINVAL, "need n_rows >= 0, row_len > 0 and at most 2^26 tokens");
  if (d->head_dim != kGdnD) return fail(STP_EUNSUPPORTED, "head_dim must be 128 (got %d)", d->head_dim);
  if (d->n_heads < 1 || d->n_heads > 64) return fail(STP_EUNSUPPORTED, "n_heads must lie in [1, 64]");
  if (!std::isfinite(d->scale)) return fail(STP_EINVAL, "scale is not finite");
  return STP_OK;
}

inline stp_status check_gdn_plan(const stp_gdn_desc* d, const int32_t* w) {
  if (!w) return fail(STP_EINVAL, "GDN plan is NULL");
  if (w[GP_MAGIC] != kGdnMagic) return fail(STP_EINVAL, "not a GDN plan (bad magic word)");
  if ((int64_t)w[GP_N] != (int64_t)d->n_rows * d->row_len)
    return fail(STP_EINVAL, "the plan covers %d tokens, the descriptor %lld", w[GP_N],
                (long long)d->n_rows * d->row_len);
  return STP_OK;
}

}  // namespace stp
