// mla_api.cu -- the C ABI of libmla_gb300 (declared in include/mla.h):
// argument validation, sizing of the decode work plan, and kernel launches
// on the caller's stream.  Allocates nothing.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdio>

#include "mla_device.cuh"

#include "params.cuh"

using namespace mla;

namespace {

constexpr int kVersion = 100;  // 0.1.0
// Largest batch * q_len * H of one call (2^26 query rows: 77 GB of absorbed
// queries alone), so that grid sizes and row indices stay within int32.
constexpr long long kMaxQueryRows = MLA_MAX_QUERY_ROWS;

std::atomic<cudaEvent_t> g_ev_start{nullptr}, g_ev_stop{nullptr};
std::atomic<int> g_inject_wait_timeout{0};
std::atomic<int> g_force_single_cta{0};

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Element code of the cache rows; 1-byte codes (INT8, FP8) carry per-token scales.
int cache_code(const mla_dims* d) {
  return d->cache_dtype == MLA_CACHE_INT8 ? kCodeInt8 : d->cache_dtype == MLA_CACHE_FP8 ? kCodeE4m3 : kCodeBf16;
}
// Bytes of per-token quantisation parameters: (scale, zero point) or a scale.
size_t scale_bytes_per_row(int code) { return code == kCodeInt8 ? 8 : code == kCodeE4m3 ? 4 : 0; }

int sm_count() {
  static std::atomic<int> cached[128];  // per device (zero-initialised)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (dev >= 0 && dev < 128 && cached[dev] > 0) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  if (dev >= 0 && dev < 128) cached[dev] = n;
  return n;
}

// Dimensions as the kernels see them for q_len query tokens per sequence:
// every (token, head) pair is one row, q_len * H rows in all.
mla_dims row_dims(const mla_dims* d, int q_len) {
  mla_dims r = *d;
  r.num_heads = d->num_heads * q_len;
  return r;
}

// The attention kernel for `rows` query rows per sequence (heads, or
// q_len x heads): more than 32 rows run on the 128-row CTA-pair kernel (any
// cache format; rows that are not a multiple of 128 pad the last group,
// which still reads each tile once where the 16/32-row kernels would read it
// once per group), except bf16 rows that make one or two 32-row groups of
// the 16/32-head CTA-pair kernel (measured on the V2-Lite batch at 4 tokens
// x 16 heads: 0.510 ms as two 32-row groups, 0.544 ms as one padded group;
// at 6 tokens 0.754 against 0.547 ms).  The rest: bf16 caches on the
// 16/32-head CTA-pair kernel, 1-byte caches (and devices that cannot place
// pairs) on single CTAs.  `units` = attention units resident at once (pairs
// or CTAs).
enum AttnKind { kAttnRows128, kAttnPair, kAttnSingle };
struct AttnChoice {
  int kind, hc, units;
};
AttnChoice choose_attention(int rows, int code) {
  const bool byte = code != kCodeBf16;
  const bool single = g_force_single_cta.load() != 0;
  const bool pair_groups = !byte && rows <= 64 && rows % 32 == 0;
  if (!single && (rows % 128 == 0 || (rows > 32 && !pair_groups))) {
    const int cap = decode_rows128_capacity(code);
    if (cap > 0) return {kAttnRows128, 128, cap};
  }
  const int hc = decode_head_group(rows, byte);
  const int pairs = byte || single ? 0 : decode_pair_capacity(hc);
  if (pairs > 0) return {kAttnPair, hc, pairs};
  return {kAttnSingle, hc, sm_count()};
}

// Automatic split count: one partition per resident attention unit of a
// head group (more partitions only add segment switches and partials to
// merge).
int effective_splits(const mla_dims* d, int num_splits) {
  if (num_splits > 0) return num_splits;
  const AttnChoice a = choose_attention(d->num_heads, cache_code(d));
  if (a.units <= 0) return -1;
  const int groups = (d->num_heads + a.hc - 1) / a.hc;
  return a.units / groups > 0 ? a.units / groups : 1;
}

int decode_rows(const mla_dims* d, const void* q_nope, const void* q_pe, const void* cache,
                const float* cache_scale_zero, int32_t num_pages, const int32_t* block_table,
                int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t batch, int32_t q_len, const void* W_UK,
                const void* W_UV, float softmax_scale, int32_t num_splits, void* workspace, size_t workspace_bytes,
                void* out, float* lse_out, mla_stream_t stream, bool reset_status);

// Append parameters shared by mla_cache_append and mla_prefill (which then
// set the token -> (sequence, position) mapping).
AppendParams append_params(const mla_dims* d, void* cache, float* cache_scale_zero, int32_t num_pages,
                           const int32_t* block_table, int32_t num_seqs, int32_t max_pages_per_seq, int32_t n_tokens,
                           const void* c_kv, const void* k_pe, double rope_theta, int32_t* device_status) {
  AppendParams p;
  p.cache = cache;
  p.scale_zero = cache_scale_zero;
  p.block_table = block_table;
  p.seq_ids = nullptr;
  p.positions = nullptr;
  p.seq_lens = nullptr;
  p.chunk = 0;
  p.c_kv = static_cast<const __nv_bfloat16*>(c_kv);
  p.k_pe = static_cast<const __nv_bfloat16*>(k_pe);
  p.status = device_status;
  p.rope_theta = rope_theta;
  // the frequencies depend only on theta: one fp64 pow per pair here instead
  // of one per token and pair on the device's slow fp64 units
  for (int i = 0; i < kRope / 2; ++i)
    p.inv_freq[i] = rope_theta > 0.0 ? std::pow(rope_theta, -double(2 * i) / double(kRope)) : 0.0;
  p.n_tokens = n_tokens;
  p.num_seqs = num_seqs;
  p.max_pages = max_pages_per_seq;
  p.num_pages = num_pages;
  p.page_size = d->page_size;
  return p;
}

}  // namespace

extern "C" {

int mla_version(void) { return kVersion; }

const char* mla_status_string(int s) {
  switch (s) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARG: return "invalid argument";
    case MLA_ERR_UNSUPPORTED: return "unsupported dimensions";
    case MLA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case MLA_ERR_CUDA: return "CUDA call failed";
    case MLA_ERR_DEVICE_TIMEOUT: return "device: bounded wait ran out";
    case MLA_ERR_DEVICE_BOUNDS: return "device: page-table entry, position or length out of range";
    default: return "unknown status";
  }
}

int mla_check_dims(const mla_dims* d) {
  if (!d) return MLA_ERR_INVALID_ARG;
  if (d->num_heads <= 0 || d->kv_lora_rank <= 0 || d->rope_dim <= 0 || d->qk_nope_dim <= 0 ||
      d->v_head_dim <= 0 || d->page_size <= 0)
    return MLA_ERR_INVALID_ARG;
  if (d->cache_dtype != MLA_CACHE_BF16 && d->cache_dtype != MLA_CACHE_INT8 && d->cache_dtype != MLA_CACHE_FP8)
    return MLA_ERR_INVALID_ARG;
  if (d->kv_lora_rank != kLatent || d->rope_dim != kRope || d->qk_nope_dim != kNope || d->v_head_dim != kVDim)
    return MLA_ERR_UNSUPPORTED;
  if (d->page_size != 16 && d->page_size != 32 && d->page_size != 64 && d->page_size != 128)
    return MLA_ERR_UNSUPPORTED;
  if (d->num_heads != 16 && d->num_heads % 32 != 0) return MLA_ERR_UNSUPPORTED;
  return MLA_OK;
}

int mla_cache_append(const mla_dims* d, void* cache, float* cache_scale_zero, int32_t num_pages,
                     const int32_t* block_table, int32_t num_seqs, int32_t max_pages_per_seq,
                     const int32_t* seq_ids, const int32_t* positions, int32_t n_tokens, const void* c_kv,
                     const void* k_pe, double rope_theta, int32_t* device_status, mla_stream_t stream) {
  int st = mla_check_dims(d);
  if (st != MLA_OK) return st;
  if (n_tokens < 0 || num_pages <= 0 || num_seqs <= 0 || max_pages_per_seq <= 0) return MLA_ERR_INVALID_ARG;
  if (n_tokens == 0) return MLA_OK;
  const int code = cache_code(d);
  const bool byte = code != kCodeBf16;
  if (!cache || !block_table || !seq_ids || !positions || !c_kv || !k_pe) return MLA_ERR_INVALID_ARG;
  if (byte && !cache_scale_zero) return MLA_ERR_INVALID_ARG;
  if (!aligned(cache, 16) || !aligned(c_kv, 16) || !aligned(k_pe, 4) || !aligned(block_table, 4) ||
      !aligned(seq_ids, 4) || !aligned(positions, 4) || (byte && !aligned(cache_scale_zero, 8)))
    return MLA_ERR_INVALID_ARG;
  AppendParams p = append_params(d, cache, cache_scale_zero, num_pages, block_table, num_seqs, max_pages_per_seq,
                                 n_tokens, c_kv, k_pe, rope_theta, device_status);
  p.seq_ids = seq_ids;
  p.positions = positions;
  return launch_append(p, code, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int mla_auto_num_splits(const mla_dims* d, int32_t batch) {
  int st = mla_check_dims(d);
  if (st != MLA_OK) return st;
  if (batch <= 0) return MLA_ERR_INVALID_ARG;
  const int s = effective_splits(d, 0);
  return s > 0 ? s : MLA_ERR_CUDA;
}

size_t mla_decode_workspace_size(const mla_dims* d, int32_t batch, int32_t num_splits) {
  return mla_decode_multi_workspace_size(d, batch, 1, num_splits);
}

size_t mla_decode_multi_workspace_size(const mla_dims* d, int32_t batch, int32_t q_len, int32_t num_splits) {
  if (q_len > MLA_MAX_Q_LEN) return 0;
  return mla_prefill_workspace_size(d, batch, q_len, num_splits);
}

size_t mla_prefill_workspace_size(const mla_dims* d, int32_t batch, int32_t chunk, int32_t num_splits) {
  if (mla_check_dims(d) != MLA_OK || batch <= 0 || num_splits < 0 || chunk < 1 || chunk > MLA_MAX_PREFILL_CHUNK)
    return 0;
  if ((long long)batch * chunk * d->num_heads > kMaxQueryRows) return 0;
  const mla_dims dr = row_dims(d, chunk);
  const int s = effective_splits(&dr, num_splits);
  if (s <= 0) return 0;
  return workspace_layout(batch, dr.num_heads, s).total;
}

int mla_decode(const mla_dims* d, const void* q_nope, const void* q_pe, const void* cache,
               const float* cache_scale_zero, int32_t num_pages, const int32_t* block_table,
               int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t batch, const void* W_UK,
               const void* W_UV, float softmax_scale, int32_t num_splits, void* workspace,
               size_t workspace_bytes, void* out, float* lse_out, mla_stream_t stream) {
  return mla_decode_multi(d, q_nope, q_pe, cache, cache_scale_zero, num_pages, block_table, max_pages_per_seq,
                          seq_lens, batch, 1, W_UK, W_UV, softmax_scale, num_splits, workspace, workspace_bytes, out,
                          lse_out, stream);
}

int mla_decode_multi(const mla_dims* d, const void* q_nope, const void* q_pe, const void* cache,
                     const float* cache_scale_zero, int32_t num_pages, const int32_t* block_table,
                     int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t batch, int32_t q_len,
                     const void* W_UK, const void* W_UV, float softmax_scale, int32_t num_splits, void* workspace,
                     size_t workspace_bytes, void* out, float* lse_out, mla_stream_t stream) {
  if (q_len > MLA_MAX_Q_LEN) return MLA_ERR_INVALID_ARG;
  return decode_rows(d, q_nope, q_pe, cache, cache_scale_zero, num_pages, block_table, max_pages_per_seq, seq_lens,
                     batch, q_len, W_UK, W_UV, softmax_scale, num_splits, workspace, workspace_bytes, out, lse_out,
                     stream, true);
}

int mla_prefill(const mla_dims* d, void* cache, float* cache_scale_zero, int32_t num_pages, const int32_t* block_table,
                int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t batch, int32_t chunk, const void* c_kv,
                const void* k_pe, double rope_theta, const void* q_nope, const void* q_pe, const void* W_UK,
                const void* W_UV, float softmax_scale, int32_t num_splits, void* workspace, size_t workspace_bytes,
                void* out, float* lse_out, mla_stream_t stream) {
  int st = mla_check_dims(d);
  if (st != MLA_OK) return st;
  if (batch <= 0 || num_pages <= 0 || max_pages_per_seq <= 0 || chunk < 1 || chunk > MLA_MAX_PREFILL_CHUNK)
    return MLA_ERR_INVALID_ARG;
  const bool byte = cache_code(d) != kCodeBf16;
  if (!cache || !block_table || !seq_lens || !c_kv || !k_pe || (byte && !cache_scale_zero)) return MLA_ERR_INVALID_ARG;
  if (!aligned(c_kv, 16) || !aligned(k_pe, 4) || (byte && !aligned(cache_scale_zero, 16)))
    return MLA_ERR_INVALID_ARG;
  if ((long long)batch * chunk > (1LL << 31) - 1) return MLA_ERR_INVALID_ARG;
  // everything decode_rows checks, before anything is launched
  const size_t need = mla_prefill_workspace_size(d, batch, chunk, num_splits);
  if (need == 0) return MLA_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return MLA_ERR_WORKSPACE;
  if (!q_nope || !q_pe || !W_UK || !W_UV || !out || !(softmax_scale > 0.f) || softmax_scale == INFINITY ||
      !aligned(cache, 16) || !aligned(q_nope, 4) || !aligned(q_pe, 4) || !aligned(W_UK, 4) || !aligned(W_UV, 4) ||
      !aligned(out, 4) || !aligned(block_table, 4) || !aligned(seq_lens, 4) || (lse_out && !aligned(lse_out, 4)))
    return MLA_ERR_INVALID_ARG;
  if ((long long)max_pages_per_seq * d->page_size > (1LL << 31) - 1) return MLA_ERR_INVALID_ARG;
  if ((long long)num_pages * d->page_size > (1LL << 31) - 1) return MLA_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the call's status word starts at MLA_OK before the append can report into it
  int* status = reinterpret_cast<int*>(static_cast<char*>(workspace) + workspace_layout(batch, d->num_heads, 1).status);
  if (cudaMemsetAsync(status, 0, sizeof(int), s) != cudaSuccess) return MLA_ERR_CUDA;
  AppendParams ap = append_params(d, cache, cache_scale_zero, num_pages, block_table, batch, max_pages_per_seq,
                                  batch * chunk, c_kv, k_pe, rope_theta, status);
  ap.seq_lens = seq_lens;
  ap.chunk = chunk;
  if (launch_append(ap, cache_code(d), s) != cudaSuccess) return MLA_ERR_CUDA;
  // the chunk's queries as multi-token rows over the cache that now holds the chunk
  return decode_rows(d, q_nope, q_pe, cache, cache_scale_zero, num_pages, block_table, max_pages_per_seq, seq_lens,
                     batch, chunk, W_UK, W_UV, softmax_scale, num_splits, workspace, workspace_bytes, out, lse_out,
                     stream, false);
}

}  // extern "C"

namespace {

// mla_decode_multi; reset_status = false leaves the status word as a kernel
// earlier in the same call (the sparse gather) set it.
int decode_rows(const mla_dims* d, const void* q_nope, const void* q_pe, const void* cache,
                const float* cache_scale_zero, int32_t num_pages, const int32_t* block_table,
                int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t batch, int32_t q_len, const void* W_UK,
                const void* W_UV, float softmax_scale, int32_t num_splits, void* workspace, size_t workspace_bytes,
                void* out, float* lse_out, mla_stream_t stream, bool reset_status) {
  int st = mla_check_dims(d);
  if (st != MLA_OK) return st;
  const int code = cache_code(d);
  const bool byte = code != kCodeBf16;
  if (batch <= 0 || num_pages <= 0 || max_pages_per_seq <= 0 || num_splits < 0) return MLA_ERR_INVALID_ARG;
  if (q_len < 1 || q_len > MLA_MAX_PREFILL_CHUNK) return MLA_ERR_INVALID_ARG;
  // query rows of the call: keeps every grid (absorption, merge) and row index in range
  if ((long long)batch * q_len * d->num_heads > kMaxQueryRows) return MLA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || softmax_scale == INFINITY) return MLA_ERR_INVALID_ARG;
  if (!q_nope || !q_pe || !cache || !block_table || !seq_lens || !W_UK || !W_UV || !out) return MLA_ERR_INVALID_ARG;
  if (byte && !cache_scale_zero) return MLA_ERR_INVALID_ARG;
  if (!aligned(cache, 16) || !aligned(q_nope, 4) || !aligned(q_pe, 4) || !aligned(W_UK, 4) || !aligned(W_UV, 4) ||
      !aligned(out, 4) || !aligned(block_table, 4) || !aligned(seq_lens, 4) || (lse_out && !aligned(lse_out, 4)) ||
      (byte && !aligned(cache_scale_zero, 16)))
    return MLA_ERR_INVALID_ARG;
  if ((long long)max_pages_per_seq * d->page_size > (1LL << 31) - 1) return MLA_ERR_INVALID_ARG;
  if ((long long)num_pages * d->page_size > (1LL << 31) - 1) return MLA_ERR_INVALID_ARG;  // row index is int32
  const mla_dims dr = row_dims(d, q_len);  // the kernels' "heads": q_len * H rows per sequence
  const int S = effective_splits(&dr, num_splits);
  if (S <= 0) return MLA_ERR_CUDA;
  const WorkspaceLayout L = workspace_layout(batch, dr.num_heads, S);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < L.total) return MLA_ERR_WORKSPACE;

  const AttnChoice attn = choose_attention(dr.num_heads, code);
  if (attn.units <= 0) return MLA_ERR_CUDA;
  const int H = dr.num_heads, hc = attn.hc, groups = (H + hc - 1) / hc;
  char* ws = static_cast<char*>(workspace);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  AbsorbParams ap;
  ap.q_nope = static_cast<const __nv_bfloat16*>(q_nope);
  ap.q_pe = static_cast<const __nv_bfloat16*>(q_pe);
  ap.W_UK = static_cast<const __nv_bfloat16*>(W_UK);
  ap.q_full = reinterpret_cast<__nv_bfloat16*>(ws + L.q_full);
  ap.q_sum = reinterpret_cast<float*>(ws + L.q_sum);
  ap.seq_lens = seq_lens;
  ap.tile_start = reinterpret_cast<int*>(ws + L.tile_start);
  ap.seg_base = reinterpret_cast<int*>(ws + L.seg_base);
  ap.len_checked = reinterpret_cast<int*>(ws + L.len_checked);
  ap.status = reinterpret_cast<int*>(ws + L.status);
  ap.batch = batch;
  ap.heads = H;
  ap.heads_w = d->num_heads;
  ap.reset_status = reset_status ? 1 : 0;
  ap.cols = batch * q_len;
  ap.max_len = max_pages_per_seq * d->page_size;
  ap.num_splits = S;
  if (launch_absorb(ap, byte, s) != cudaSuccess) return MLA_ERR_CUDA;

  DecodeParams dp;
  dp.q_full = ap.q_full;
  dp.q_sum = ap.q_sum;
  dp.cache = cache;
  dp.scale_zero = cache_scale_zero;
  dp.block_table = block_table;
  dp.tile_start = ap.tile_start;
  dp.seg_base = ap.seg_base;
  dp.len = ap.len_checked;
  dp.partial_o = reinterpret_cast<float*>(ws + L.partial_o);
  dp.partial_lse = reinterpret_cast<float*>(ws + L.partial_lse);
  dp.status = ap.status;
  dp.batch = batch;
  dp.heads = H;
  dp.head_group = hc;
  dp.num_groups = groups;
  dp.page_size = d->page_size;
  dp.max_pages = max_pages_per_seq;
  dp.num_pages = num_pages;
  dp.num_splits = S;
  dp.q_len = q_len;
  dp.heads_w = d->num_heads;
  dp.scale_log2 = softmax_scale * kLog2e;
  dp.inject_wait_timeout = g_inject_wait_timeout.load();
  const int per_group = attn.units / groups > 0 ? attn.units / groups : 1;
  const int per_group_used = S < per_group ? S : per_group;
  cudaEvent_t ev0 = g_ev_start.load(), ev1 = g_ev_stop.load();
  if (ev0 && ev1 && cudaEventRecord(ev0, s) != cudaSuccess) return MLA_ERR_CUDA;
  const cudaError_t le = attn.kind == kAttnRows128 ? launch_decode_rows128(dp, code, per_group_used, s)
                         : attn.kind == kAttnPair  ? launch_decode_pair(dp, hc, per_group_used, s)
                                                   : launch_decode_tc(dp, hc, code, per_group_used * groups, s);
  if (le != cudaSuccess) return MLA_ERR_CUDA;
  if (ev0 && ev1 && cudaEventRecord(ev1, s) != cudaSuccess) return MLA_ERR_CUDA;

  CombineUVParams cp;
  cp.partial_o = dp.partial_o;
  cp.partial_lse = dp.partial_lse;
  cp.seg_base = dp.seg_base;
  cp.status = dp.status;
  cp.sm_count = sm_count();
  cp.W_UV = static_cast<const __nv_bfloat16*>(W_UV);
  cp.out = static_cast<__nv_bfloat16*>(out);
  cp.lse_out = lse_out;
  cp.batch = batch;
  cp.heads = H;
  cp.heads_w = d->num_heads;
  cp.q_len = q_len;
  if (launch_combine_uv(cp, s) != cudaSuccess) return MLA_ERR_CUDA;
  return MLA_OK;
}

// Workspace of mla_decode_sparse: the decode's own workspace first (so that
// the call's status word is the workspace's first 4 bytes), then the
// gathered cache [batch * pps pages, P, 576] (+ per-token scales), its page
// table [batch, pps] and lengths [batch]; pps = ceil(top_k / P).
struct SparseLayout {
  size_t decode, cache, scale_zero, table, lens, total;
  int pps;
};

SparseLayout sparse_layout(const mla_dims* d, int batch, int top_k, size_t decode_bytes) {
  SparseLayout L;
  const int code = cache_code(d);
  L.pps = (top_k + d->page_size - 1) / d->page_size;
  const size_t rows = size_t(batch) * L.pps * d->page_size;
  size_t off = 0;
  L.decode = off;      off = align256(off + decode_bytes);
  L.cache = off;       off = align256(off + rows * (code == kCodeBf16 ? 1152 : 576));
  L.scale_zero = off;  off = align256(off + rows * scale_bytes_per_row(code));
  L.table = off;       off = align256(off + size_t(batch) * L.pps * 4);
  L.lens = off;        off = align256(off + size_t(batch) * 4);
  L.total = off;
  return L;
}

}  // namespace

extern "C" {

size_t mla_decode_sparse_workspace_size(const mla_dims* d, int32_t batch, int32_t top_k, int32_t num_splits) {
  if (top_k < 1 || top_k > MLA_MAX_TOP_K) return 0;
  const size_t dec = mla_decode_workspace_size(d, batch, num_splits);
  if (dec == 0) return 0;
  return sparse_layout(d, batch, top_k, dec).total;
}

int mla_decode_sparse(const mla_dims* d, const void* q_nope, const void* q_pe, const void* cache,
                      const float* cache_scale_zero, int32_t num_pages, const int32_t* block_table,
                      int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t batch,
                      const int32_t* token_indices, int32_t top_k, const void* W_UK, const void* W_UV,
                      float softmax_scale, int32_t num_splits, void* workspace, size_t workspace_bytes, void* out,
                      float* lse_out, mla_stream_t stream) {
  int st = mla_check_dims(d);
  if (st != MLA_OK) return st;
  const int code = cache_code(d);
  const bool byte = code != kCodeBf16;
  if (batch <= 0 || num_pages <= 0 || max_pages_per_seq <= 0 || num_splits < 0) return MLA_ERR_INVALID_ARG;
  if (top_k < 1 || top_k > MLA_MAX_TOP_K || !token_indices || !aligned(token_indices, 4)) return MLA_ERR_INVALID_ARG;
  if (!cache || !block_table || !seq_lens || (byte && !cache_scale_zero)) return MLA_ERR_INVALID_ARG;
  if (!aligned(cache, 16) || !aligned(block_table, 4) || !aligned(seq_lens, 4) ||
      (byte && !aligned(cache_scale_zero, 8)))
    return MLA_ERR_INVALID_ARG;
  if ((long long)max_pages_per_seq * d->page_size > (1LL << 31) - 1) return MLA_ERR_INVALID_ARG;
  if ((long long)num_pages * d->page_size > (1LL << 31) - 1) return MLA_ERR_INVALID_ARG;
  const size_t dec = mla_decode_workspace_size(d, batch, num_splits);
  if (dec == 0) return MLA_ERR_CUDA;
  const SparseLayout L = sparse_layout(d, batch, top_k, dec);
  if ((long long)batch * L.pps * d->page_size > (1LL << 31) - 1) return MLA_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < L.total) return MLA_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the call's status word starts at MLA_OK before the gather can report into it
  int* status = reinterpret_cast<int*>(ws + L.decode + workspace_layout(batch, d->num_heads, 1).status);
  if (cudaMemsetAsync(status, 0, sizeof(int), s) != cudaSuccess) return MLA_ERR_CUDA;
  GatherParams gp;
  gp.cache = cache;
  gp.scale_zero = cache_scale_zero;
  gp.block_table = block_table;
  gp.seq_lens = seq_lens;
  gp.indices = token_indices;
  gp.out_cache = ws + L.cache;
  gp.out_scale_zero = byte ? reinterpret_cast<float*>(ws + L.scale_zero) : nullptr;
  gp.out_table = reinterpret_cast<int*>(ws + L.table);
  gp.out_lens = reinterpret_cast<int*>(ws + L.lens);
  gp.status = status;
  gp.batch = batch;
  gp.top_k = top_k;
  gp.max_pages = max_pages_per_seq;
  gp.num_pages = num_pages;
  gp.page_size = d->page_size;
  gp.pages_per_seq = L.pps;
  if (launch_gather(gp, code, s) != cudaSuccess) return MLA_ERR_CUDA;
  // the dense decode over the gathered rows, with the lengths the gather wrote
  return decode_rows(d, q_nope, q_pe, gp.out_cache, gp.out_scale_zero, batch * L.pps, gp.out_table, L.pps,
                     gp.out_lens, batch, 1, W_UK, W_UV, softmax_scale, num_splits, ws + L.decode, dec, out, lse_out,
                     stream, false);
}

int mla_combine(const mla_dims* d, const float* partial_o, const float* partial_lse, int32_t batch,
                int32_t num_splits, float* o_lat_out, float* lse_out, mla_stream_t stream) {
  int st = mla_check_dims(d);
  if (st != MLA_OK) return st;
  if (batch <= 0 || num_splits <= 0) return MLA_ERR_INVALID_ARG;
  if (!partial_o || !partial_lse || !o_lat_out) return MLA_ERR_INVALID_ARG;
  if (!aligned(partial_o, 4) || !aligned(partial_lse, 4) || !aligned(o_lat_out, 4) || (lse_out && !aligned(lse_out, 4)))
    return MLA_ERR_INVALID_ARG;
  CombineParams p;
  p.partial_o = partial_o;
  p.partial_lse = partial_lse;
  p.o_lat = o_lat_out;
  p.lse_out = lse_out;
  p.batch = batch;
  p.splits = num_splits;
  p.heads = d->num_heads;
  p.dim = d->kv_lora_rank;
  return launch_combine(p, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int mla_read_status_word(const int32_t* device_status, int32_t* status_out, mla_stream_t stream) {
  if (!device_status || !status_out) return MLA_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MLA_ERR_CUDA;
  if (cudaMemcpy(status_out, device_status, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

int mla_read_device_status(const void* workspace, int32_t* status_out, mla_stream_t stream) {
  if (!workspace) return MLA_ERR_INVALID_ARG;
  return mla_read_status_word(static_cast<const int32_t*>(workspace), status_out, stream);
}

int mla_test_force_single_cta(int32_t enable) {
  g_force_single_cta.store(enable != 0);
  return MLA_OK;
}

int mla_test_inject_wait_timeout(int32_t enable) {
  g_inject_wait_timeout.store(enable != 0);
  return MLA_OK;
}

int mla_set_timing_events(mla_event_t start, mla_event_t stop) {
  if ((start == nullptr) != (stop == nullptr)) return MLA_ERR_INVALID_ARG;
  g_ev_start.store(reinterpret_cast<cudaEvent_t>(start));
  g_ev_stop.store(reinterpret_cast<cudaEvent_t>(stop));
  return MLA_OK;
}

}  // extern "C"
