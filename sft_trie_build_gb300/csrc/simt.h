// Arguments shared by the tree-attention launchers of libstp.so.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace stp {

struct AttnArgs {
  int R, T, Hq, Hkv, D;
  float scale;
  const void* q;
  const void* k;
  const void* v;
  const void* o_in;      // forward output (backward only)
  const void* dout;      // dO (backward only)
  void* o;               // forward output
  float* lse;            // [R, Hq, T]
  void* dq;
  void* dk;
  void* dv;
  const int32_t* se;     // subtree_end [R, T]
  const int32_t* csr_cnt;
  const int32_t* csr;
  const int32_t* csc_cnt;
  const int32_t* csc;
  const int32_t* csr_off;   // pair numbering of stp_classify (tile_meta)
  const int32_t* row_base;
  const int32_t* csc_pair;
  float* delta;          // [R, Hq, T] (backward, fp32 path): Delta
  void* sbias;           // [R, Hq, NT] bias tiles of the scores (backward, bf16 path)
  void* dbias;           // [R, Hq, NT] bias tiles of dP (backward, bf16 path)
  void* ds;              // dS^T tile slots (backward, bf16 path)
  int64_t ds_cap;        // pairs a slot holds
  int ds_slots;          // slots (kv-head groups whose tiles are held at once)
  size_t ds_slot_bytes;  // bytes per slot
  uint32_t* err;         // device error word of the workspace
};

cudaError_t simt_fwd(const AttnArgs& a, bool bf16, cudaStream_t s);
cudaError_t simt_bwd(const AttnArgs& a, bool bf16, cudaStream_t s);

}  // namespace stp
