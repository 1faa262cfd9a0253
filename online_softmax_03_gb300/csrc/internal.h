// internal.h -- declarations shared by the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace attn_host {

struct PrefillArgs {
  const void *q, *k, *v;
  void *o;
  float *lse;
  int B, Hq, Hkv, Tq, Tk, d, causal;
  int window;  // > 0: causal sliding window of this many keys (0 = none)
  float scale;
  cudaStream_t stream;
  unsigned long long wait_ns;
  int inject;
  // packed variable-length batches: q [total_q, Hq, d], k/v [total_k, Hkv, d],
  // sequence b at cu_q[b]..cu_q[b+1] / cu_k[b]..cu_k[b+1]; B = sequences,
  // Tq / Tk = the longest query / key sequence allowed
  bool varlen = false;
  const int *cu_q = nullptr, *cu_k = nullptr;
  int total_q = 0, total_k = 0;
  void *workspace = nullptr;
  size_t workspace_bytes = 0;
};

struct DecodeArgs {
  const void *q, *k, *v;
  void *o;
  float *lse;
  int B, Hq, Hkv, Tk, d;  // paged: Tk = the longest allowed sequence
  float scale;
  void *workspace;
  size_t workspace_bytes;
  cudaStream_t stream;
  unsigned long long wait_ns;
  int inject = 0;  // test hook (attn_debug_set)
  // paged cache (k, v are page pools [num_pages, Hkv, page_size, d])
  bool paged = false;
  const int *block_table = nullptr;
  const int *seq_lens = nullptr;
  int page_size = 0, num_pages = 0, max_pages = 0;
};

struct BwdArgs {
  const void *q, *k, *v, *o, *dout;
  const float *lse;
  void *dq, *dk, *dv;
  int B, Hq, Hkv, Tq, Tk, d, causal;
  int window = 0;  // > 0: causal sliding window of this many keys
  float scale;
  void *workspace;
  size_t workspace_bytes;
  cudaStream_t stream;
  unsigned long long wait_ns;
  int inject = 0;  // test hook (attn_debug_set)
};

// Return an attn_status code.
int prefill_launch(const PrefillArgs &a);
int decode_launch(const DecodeArgs &a);
int prefill_take_status(cudaStream_t s, unsigned int *out);
int decode_take_status(cudaStream_t s, unsigned int *out);
int bwd_launch(const BwdArgs &a);
int bwd_take_status(cudaStream_t s, unsigned int *out);
size_t bwd_workspace_bytes_for(int B, int Hq, int Tq, int d);

// Shared helpers (api.cu).
int validate_decode_args(const void *q, const void *k, const void *v, const void *o,
                         const float *lse, int B, int Hq, int Hkv, int Tk, int d,
                         float scale, float *scale_out);
// Compute capability 10.3 check and SM count of the current device, queried
// once per device and cached.
int check_device_sm103(int *num_sms);
// Device address of a __device__ symbol (the address of its host-side
// stand-in) on the current device, looked up once per (symbol, device).
int symbol_address(const void *symbol, void **out);
// Raises a kernel's dynamic shared-memory limit to `bytes`, once per
// (kernel, device).
int ensure_smem_limit(const void *kern, int bytes);
// The wait limit attn_debug_set chose (1 s unless a test changed it).
unsigned long long wait_limit_ns();
// The test hook attn_debug_set chose (0 = none).
int inject_hook();
// 3-D bf16 tensor map over a dense (inner, rows, planes) array; the box is
// box_inner x box_rows x box_planes elements.
bool encode_tmap_3d_bf16(CUtensorMap *map, const void *base, uint64_t inner,
                         uint64_t rows, uint64_t planes, uint32_t box_inner,
                         uint32_t box_rows, uint32_t box_planes, int swizzle_bytes);

// The same for a 3-D fp32 tensor map with 128-byte swizzle (box_inner = 32).
bool encode_tmap_3d_f32(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows,
                        uint64_t planes, uint32_t box_inner, uint32_t box_rows,
                        uint32_t box_planes);

// Packed-batch planning list capacity and its scratch bytes.
long long varlen_list_capacity(int B, int total_q, int max_seqlen_q);
size_t varlen_workspace_bytes_for(int B, int total_q, int max_seqlen_q);

// Decode split plan: depends only on sizes (and the SM count for the chosen
// split, bounded above by the size-only maximum).
int decode_max_splits(int Tk);
size_t decode_workspace_bytes_for(int B, int Hq, int Tk, int d);

}  // namespace attn_host
