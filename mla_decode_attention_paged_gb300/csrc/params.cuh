// params.cuh -- parameter blocks passed from the host ABI to the kernels,
// and the launch functions of each kernel file.
#pragma once

#include <utility>

#include "mla_device.cuh"

namespace mla {

// Element type of the cached rows (mla_cache_dtype): bf16 values, INT8 codes
// with a per-token (scale, zero point), or FP8 E4M3 codes with a per-token
// scale.
enum CacheCode : int { kCodeBf16 = 0, kCodeInt8 = 1, kCodeE4m3 = 2 };

// Multi-token decode (q_len query tokens per sequence) runs the same kernels
// over "rows": row v = t * heads_w + h of a sequence is query token t, head
// h.  `heads` below counts rows (q_len * heads_w); the weights have heads_w
// heads and row v uses head v % heads_w.
struct AbsorbParams {
  const __nv_bfloat16* q_nope;  // [B, heads, 128]
  const __nv_bfloat16* q_pe;    // [B, heads, 64]
  const __nv_bfloat16* W_UK;    // [heads_w, 128, 512]
  __nv_bfloat16* q_full;        // [B, H, 576] (fp16 bit patterns for 1-byte caches)
  float* q_sum;                 // [B, H, kQSumParts]
  // plan
  const int* seq_lens;
  int* tile_start;
  int* seg_base;
  int* len_checked;
  int* status;
  int batch, heads, heads_w, max_len, num_splits;
  int reset_status;  // 1: the plan starts the call's status word at MLA_OK (0: a kernel before it did)
  // The absorption GEMM's view of the rows: row v = t * heads_w + h of
  // sequence b is column b * q_len + t of weight head h, so each head's
  // product covers every (sequence, token) column at once; cols = batch *
  // q_len, q_nope / q_full / q_sum rows are at (column * heads_w + h).
  int cols;
};

// Sparse (top-k) decode: the listed rows of each sequence, compacted in list
// order into pages_per_seq pages of the gathered cache (sequence b owns pages
// [b pages_per_seq, (b + 1) pages_per_seq)), its length and page-table row.
struct GatherParams {
  const void* cache;         // bf16, int8 or e4m3 [num_pages, P, 576]
  const float* scale_zero;   // [num_pages, P, 2] (INT8) or [num_pages, P] (FP8)
  const int* block_table;    // [B, max_pages]
  const int* seq_lens;       // [B]
  const int* indices;        // [B, top_k], -1 = padding
  void* out_cache;           // [B * pages_per_seq, P, 576]
  float* out_scale_zero;     // [B * pages_per_seq, P, 2] (INT8) or [.., P] (FP8)
  int* out_table;            // [B, pages_per_seq]
  int* out_lens;             // [B]
  int* status;               // MLA_ERR_DEVICE_BOUNDS for bad entries (zeroed on the stream before the launch)
  int batch, top_k, max_pages, num_pages, page_size, pages_per_seq;
};

struct AppendParams {
  void* cache;                   // bf16, int8 or e4m3 [num_pages, P, 576]
  float* scale_zero;             // [num_pages, P, 2] (INT8) or [num_pages, P] (FP8)
  const int* block_table;        // [num_seqs, max_pages]
  const int* seq_ids;            // [N]   (chunk == 0)
  const int* positions;          // [N]   (chunk == 0)
  const int* seq_lens;           // [num_seqs] (chunk > 0: token i is token i % chunk of sequence
                                 // i / chunk, at position seq_lens[b] - chunk + i % chunk)
  int chunk;                     // 0: explicit seq_ids / positions; > 0: prefill chunk per sequence
  const __nv_bfloat16* c_kv;     // [N, 512]
  const __nv_bfloat16* k_pe;     // [N, 64]
  int* status;                   // optional
  double rope_theta;
  double inv_freq[kRope / 2];    // theta^(-2i/64), evaluated on the host in fp64
  int n_tokens, num_seqs, max_pages, num_pages, page_size;
};

struct CombineUVParams {
  const float* partial_o;     // [NSEG, H, 512]
  const float* partial_lse;   // [NSEG, H]
  const int* seg_base;        // [B + 1]
  const __nv_bfloat16* W_UV;  // [heads_w, 128, 512]
  __nv_bfloat16* out;         // [B, heads, 128]
  float* lse_out;             // [B, heads] or null
  int* status;
  int batch, heads, heads_w;
  int q_len;                  // rows per sequence = q_len * heads_w; column c = b * q_len + t
  int sm_count;               // sizes the grid
};

struct CombineParams {
  const float* partial_o;    // [B, S, H, D]
  const float* partial_lse;  // [B, S, H]
  float* o_lat;              // [B, H, D]
  float* lse_out;            // [B, H] or null
  int batch, splits, heads, dim;
};

cudaError_t launch_absorb(const AbsorbParams& p, bool fp16_out, cudaStream_t stream);
cudaError_t launch_append(const AppendParams& p, int code, cudaStream_t stream);
cudaError_t launch_combine_uv(const CombineUVParams& p, cudaStream_t stream);
cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream);
cudaError_t launch_gather(const GatherParams& p, int code, cudaStream_t stream);
cudaError_t launch_decode_tc(const DecodeParams& p, int hc, int code, int grid, cudaStream_t stream);
int decode_head_group(int heads, bool byte_cache);
// Launches `kernel` with programmatic dependent launch (and, if cluster_x > 1,
// thread-block clusters of cluster_x CTAs).  The kernels of the decode step
// (append, absorb, attention, merge + up-projection) set up their shared
// memory, barriers and tensor memory, then call griddep_wait() before their
// first global-memory access and griddep_launch_dependents() after it, so
// each launch and prologue overlaps the tail of the kernel before it.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[2];
  unsigned n = 0;
  at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 1) {
    at[n].id = cudaLaunchAttributeClusterDimension;
    at[n].val.clusterDim.x = cluster_x;
    at[n].val.clusterDim.y = 1;
    at[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = at;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// bf16 caches: CTA-cluster kernel.  Capacity = clusters resident at once (0 if none).
int decode_pair_capacity(int hc);
cudaError_t launch_decode_pair(const DecodeParams& p, int hc, int clusters_per_group, cudaStream_t stream);
// Groups of 128 query rows, any cache format (CacheCode): CTA-pair kernel
// with the rows on the MMA's M extent.  Capacity = pairs resident at once (0 if none).
int decode_rows128_capacity(int code);
cudaError_t launch_decode_rows128(const DecodeParams& p, int code, int clusters_per_group, cudaStream_t stream);

}  // namespace mla
