// params.cuh -- parameter blocks passed from the host ABI to the kernels,
// and the launch functions of each kernel file.
#pragma once

#include "mla_device.cuh"

namespace mla {

struct AbsorbParams {
  const __nv_bfloat16* q_nope;  // [B, H, 128]
  const __nv_bfloat16* q_pe;    // [B, H, 64]
  const __nv_bfloat16* W_UK;    // [H, 128, 512]
  __nv_bfloat16* q_full;        // [B, H, 576] (fp16 bit patterns for INT8 caches)
  float* q_sum;                 // [B, H, kQSumParts]
  // plan
  const int* seq_lens;
  int* tile_start;
  int* seg_base;
  int* len_checked;
  int* status;
  int batch, heads, max_len, num_splits;
};

struct AppendParams {
  void* cache;                   // bf16 or int8 [num_pages, P, 576]
  float* scale_zero;             // [num_pages, P, 2] (INT8)
  const int* block_table;        // [num_seqs, max_pages]
  const int* seq_ids;            // [N]
  const int* positions;          // [N]
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
  float* o_lat;               // [B, H, 512] merged latent outputs (written by the merge kernel)
  const __nv_bfloat16* W_UV;  // [H, 128, 512]
  __nv_bfloat16* out;         // [B, H, 128]
  float* lse_out;             // [B, H] or null
  int batch, heads;
  int max_segments;           // num_splits + batch: bound on the segments of all sequences
};

struct CombineParams {
  const float* partial_o;    // [B, S, H, D]
  const float* partial_lse;  // [B, S, H]
  float* o_lat;              // [B, H, D]
  float* lse_out;            // [B, H] or null
  int batch, splits, heads, dim;
};

cudaError_t launch_absorb(const AbsorbParams& p, bool fp16_out, cudaStream_t stream);
cudaError_t launch_append(const AppendParams& p, bool int8, cudaStream_t stream);
cudaError_t launch_combine_uv(const CombineUVParams& p, cudaStream_t stream);
cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream);
cudaError_t launch_decode_tc(const DecodeParams& p, int hc, bool int8, int grid, cudaStream_t stream);
int decode_head_group(int heads, bool int8);
// bf16 caches: CTA-pair kernel.  Capacity = clusters of two resident at once (0 if none).
int decode_pair_capacity(int hc);
cudaError_t launch_decode_pair(const DecodeParams& p, int hc, int pairs_per_group, cudaStream_t stream);

}  // namespace mla
