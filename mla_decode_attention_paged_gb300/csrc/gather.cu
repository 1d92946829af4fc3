// gather.cu -- sparse (top-k) decode: the selected cached rows of every
// sequence, compacted into a small paged cache that the dense decode then
// reads ("Seven Ways LLMs Handle Attention", section 6, "Sparse attention:
// keep every token, read only some": the full cache stays, and each new token
// attends only to the top-k tokens an indexer picked -- the indexer is not
// part of this path).
//
// Entry i of sequence b names cache position indices[b][i]; -1 is padding.
// The valid entries keep their list order: entry i goes to row
// (number of valid entries before i) of sequence b's gathered pages, so the
// dense decode over the gathered rows attends to exactly the listed tokens.
// Positions outside [0, seq_len) (and lengths outside the page table) are
// reported as MLA_ERR_DEVICE_BOUNDS and skipped.
#include "blackwell_ptx.cuh"
#include "params.cuh"

namespace mla {

constexpr int kGatherEntries = 64;   // list entries per CTA
constexpr int kGatherThreads = 256;  // 8 warps; a warp copies one row at a time

template <int kCode>
__global__ void __launch_bounds__(kGatherThreads) gather_kernel(GatherParams p) {
  __shared__ int cnt[kGatherThreads / 32];   // per warp: valid entries before the chunk
  __shared__ int chunk_cnt[kGatherEntries / 32];  // per warp of the chunk: its valid entries
  __shared__ int dest[kGatherEntries];
  __shared__ int srow[kGatherEntries];
  __shared__ int before_total;
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const int b = blockIdx.y, e0 = blockIdx.x * kGatherEntries, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int P = p.page_size;
  int L = p.seq_lens[b];
  if (L < 0 || L > p.max_pages * P) {
    if (blockIdx.x == 0 && tid == 0) set_status(p.status, MLA_ERR_DEVICE_BOUNDS);
    L = 0;
  }
  const int* idx = p.indices + size_t(b) * p.top_k;
  // valid entries before this CTA's chunk
  int c = 0;
  for (int i = tid; i < e0; i += kGatherThreads) {
    const int v = idx[i];
    c += v >= 0 && v < L;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  if (lane == 0) cnt[warp] = c;
  __syncthreads();
  if (tid == 0) {
    int s = 0;
    for (int w = 0; w < kGatherThreads / 32; ++w) s += cnt[w];
    before_total = s;
  }
  // this chunk: destination row of each valid entry (list order), source row
  if (tid < kGatherEntries) {
    const int i = e0 + tid;
    const int v = i < p.top_k ? idx[i] : -1;
    bool ok = v >= 0 && v < L;
    if (i < p.top_k && !ok && v != -1) set_status(p.status, MLA_ERR_DEVICE_BOUNDS);
    int page = -1;
    if (ok) {
      page = p.block_table[size_t(b) * p.max_pages + v / P];
      if (page < 0 || page >= p.num_pages) {
        set_status(p.status, MLA_ERR_DEVICE_BOUNDS);
        ok = false;
      }
    }
    const unsigned m = __ballot_sync(0xffffffffu, ok);  // tid < 64: warps 0 and 1, whole warps
    const int rank_in_warp = __popc(m & ((1u << lane) - 1));
    if (lane == 0) chunk_cnt[warp] = __popc(m);
    dest[tid] = ok ? rank_in_warp : -1;
    srow[tid] = ok ? page * P + v % P : 0;
  }
  __syncthreads();
  if (tid < kGatherEntries && dest[tid] >= 0) dest[tid] += before_total + (tid >= 32 ? chunk_cnt[0] : 0);
  __syncthreads();
  // copy the rows: warp w takes entries w, w + 8, ...
  const size_t base_row = size_t(b) * p.pages_per_seq * P;
  constexpr int kRowBytes = kCode == kCodeBf16 ? 1152 : 576, kPieces = kRowBytes / 16;
  for (int e = warp; e < kGatherEntries; e += kGatherThreads / 32) {
    const int d = dest[e];
    if (d < 0) continue;
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.cache) + size_t(srow[e]) * kRowBytes);
    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out_cache) + (base_row + d) * kRowBytes);
    for (int q = lane; q < kPieces; q += 32) dst[q] = src[q];
    if (kCode == kCodeInt8 && lane == 0)
      reinterpret_cast<float2*>(p.out_scale_zero)[base_row + d] = reinterpret_cast<const float2*>(p.scale_zero)[srow[e]];
    if (kCode == kCodeE4m3 && lane == 0) p.out_scale_zero[base_row + d] = p.scale_zero[srow[e]];
  }
  // the last chunk of a sequence writes its length and page-table row
  if (blockIdx.x == gridDim.x - 1) {
    if (tid == 0) p.out_lens[b] = before_total + chunk_cnt[0] + chunk_cnt[1];
    for (int j = tid; j < p.pages_per_seq; j += kGatherThreads) p.out_table[size_t(b) * p.pages_per_seq + j] = b * p.pages_per_seq + j;
  }
}

cudaError_t launch_gather(const GatherParams& p, int code, cudaStream_t stream) {
  const dim3 grid((p.top_k + kGatherEntries - 1) / kGatherEntries, p.batch);
  if (code == kCodeInt8) return launch_pdl(gather_kernel<kCodeInt8>, grid, dim3(kGatherThreads), 0, stream, 1, p);
  if (code == kCodeE4m3) return launch_pdl(gather_kernel<kCodeE4m3>, grid, dim3(kGatherThreads), 0, stream, 1, p);
  return launch_pdl(gather_kernel<kCodeBf16>, grid, dim3(kGatherThreads), 0, stream, 1, p);
}

}  // namespace mla
