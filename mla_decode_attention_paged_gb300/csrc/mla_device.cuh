// mla_device.cuh -- shared device-side definitions of libmla_gb300: sizes,
// the decode work plan (how the batch's KV tiles are cut into partitions and
// per-sequence segments), and small helpers.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/mla.h"

namespace mla {

constexpr int kLatent = 512;           // d_c
constexpr int kRope = 64;              // d_rope
constexpr int kRow = kLatent + kRope;  // 576 numbers per token per layer
constexpr int kNope = 128;             // per-head content query width
constexpr int kVDim = 128;             // per-head value width
constexpr int kQSumParts = 8;          // q_sum partials per (sequence, head)
constexpr int kTile = 128;             // tokens per decode tile (one MMA M extent)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Workspace layout of mla_decode (all offsets 256-byte aligned):
//   [0]            int32 status word, int32 effective split count (+ padding)
//   tile_start     int32 [B + 1]   prefix sum of ceil(len_b / kTile)
//   seg_base       int32 [B + 1]   prefix sum of the number of segments per sequence
//   len_checked    int32 [B]       seq_lens after range checks (0 if rejected)
//   q_full         bf16  [B, H, 576]  [W^UK_h^T q_nope | q_pe] per (b, h)
//   q_sum          fp32  [B, H, 8]    partial sums of q_full's 576 values (INT8 caches):
//                                     part c covers latent dims [64c, 64c + 64), part 0 also the RoPE part
//   partial_lse    fp32  [NSEG, H]
//   partial_o      fp32  [NSEG, H, 512]   NSEG = num_splits + B (upper bound)
struct WorkspaceLayout {
  size_t status, tile_start, seg_base, len_checked, q_full, q_sum, partial_lse, partial_o, total;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

__host__ __device__ inline WorkspaceLayout workspace_layout(int batch, int heads, int num_splits) {
  WorkspaceLayout L;
  size_t off = 0;
  L.status = off;       off = align256(off + 4);
  L.tile_start = off;   off = align256(off + 4 * size_t(batch + 1));
  L.seg_base = off;     off = align256(off + 4 * size_t(batch + 1));
  L.len_checked = off;  off = align256(off + 4 * size_t(batch));
  L.q_full = off;       off = align256(off + 2 * size_t(batch) * heads * kRow);
  L.q_sum = off;        off = align256(off + 4 * size_t(batch) * heads * kQSumParts);
  const size_t nseg = size_t(num_splits) + batch;
  L.partial_lse = off;  off = align256(off + 4 * nseg * heads);
  L.partial_o = off;    off = align256(off + 4 * nseg * heads * kLatent);
  L.total = off;
  return L;
}

// ----- work plan ------------------------------------------------------------
// Each head group's work is the list of (sequence, tile) units in sequence
// order, W units in all.  It is cut into S partitions of (nearly) equal size:
// partition p holds units [floor(p*W/S), floor((p+1)*W/S)).  A segment is the
// part of one sequence inside one partition; each segment yields one partial
// result (normalised latent output + log-sum-exp), merged later by LSE.
__host__ __device__ inline long long part_start(long long p, long long W, long long S) {
  return (p * W) / S;
}
// The partition holding unit x (0 <= x < W): the largest p with part_start(p) <= x.
__host__ __device__ inline long long part_of(long long x, long long W, long long S) {
  return ((x + 1) * S - 1) / W;
}

struct TileInfo {
  int b;        // sequence
  int tile;     // tile index within the sequence
  int valid;    // valid tokens in this tile (1..128)
  int seg;      // segment (partial-result) index
  bool first;   // first tile of its segment
  bool last;    // last tile of its segment
};

// The plan kernel stores S_eff = min(num_splits, W) next to the status word,
// so that every partition is non-empty (partition starts strictly increase)
// and the segments of a sequence are exactly the partitions its tiles touch.
// Walks the units of one CTA: partitions [pa, pb) of the list.
//
// kInline = false keeps the rare paths (init and the boundary crossings, which
// hold the 64-bit divisions) out of line so that each warp role's copy of the
// walker stays small where instruction-cache space is tight; their `this`
// argument then puts the walker in local memory, which every tile's next()
// reads and writes.  kInline = true inlines everything, and the walker lives
// in registers (the CTA-pair kernel: 2.7% faster on V2-Lite; the single-CTA
// kernel's larger code runs slower that way).
template <bool kInline>
struct TileWalkerT {
  const int* tile_start;
  const int* seg_base;
  const int* len;
  long long W, S, u, u_end;
  long long p, p_start, p_next;  // current partition and its units [p_start, p_next)
  long long s_b, e_b;            // units of sequence b: [s_b, e_b)
  int b, len_b, seg_b;           // seg_b = first segment of sequence b minus its first partition

  __device__ __forceinline__ void init_body(const int* ts, const int* sb, const int* ln, int batch, int num_splits,
                                            long long pa, long long pb) {
    tile_start = ts;
    seg_base = sb;
    len = ln;
    W = ts[batch];
    S = num_splits;
    u = part_start(pa, W, S);
    u_end = part_start(pb, W, S);
    p = pa;
    p_start = u;
    p_next = part_start(pa + 1, W, S);
    // first sequence whose tiles reach past u (binary search over tile_start)
    int lo = 0, hi = batch;  // answer in [0, batch)
    while (lo < hi) {
      int mid = (lo + hi) >> 1;
      if (ts[mid + 1] <= u) lo = mid + 1; else hi = mid;
    }
    b = lo;
    enter_sequence_body();
  }
  __device__ __forceinline__ void enter_sequence_body() {
    s_b = tile_start[b];
    e_b = tile_start[b + 1];
    len_b = len[b];
    seg_b = seg_base[b] - int(part_of(s_b, W, S));
  }
  __device__ __forceinline__ void enter_partition_body() {
    while (p_next <= u) {
      ++p;
      p_start = p_next;
      p_next = part_start(p + 1, W, S);
    }
  }
  __device__ __noinline__ void init_out_of_line(const int* ts, const int* sb, const int* ln, int batch,
                                                int num_splits, long long pa, long long pb) {
    init_body(ts, sb, ln, batch, num_splits, pa, pb);
  }
  __device__ __noinline__ void enter_sequence_out_of_line() { enter_sequence_body(); }
  __device__ __noinline__ void enter_partition_out_of_line() { enter_partition_body(); }

  __device__ __forceinline__ void init(const int* ts, const int* sb, const int* ln, int batch, int num_splits,
                                       long long pa, long long pb) {
    if constexpr (kInline) init_body(ts, sb, ln, batch, num_splits, pa, pb);
    else init_out_of_line(ts, sb, ln, batch, num_splits, pa, pb);
  }

  // Divisions only when a partition boundary is crossed; the plan's
  // arrays are read only when a sequence boundary is.
  __device__ __forceinline__ bool next(TileInfo& t) {
    if (u >= u_end) return false;
    if (e_b <= u) {
      do ++b; while (tile_start[b + 1] <= u);
      if constexpr (kInline) enter_sequence_body();
      else enter_sequence_out_of_line();
    }
    if (p_next <= u) {
      if constexpr (kInline) enter_partition_body();
      else enter_partition_out_of_line();
    }
    t.b = b;
    t.tile = int(u - s_b);
    const int v = len_b - t.tile * kTile;
    t.valid = v > kTile ? kTile : v;
    t.first = (u == s_b) || (u == p_start);
    t.last = (u + 1 == e_b) || (u + 1 == p_next);
    t.seg = seg_b + int(p);
    ++u;
    return true;
  }
};
using TileWalker = TileWalkerT<false>;

struct DecodeParams {
  const __nv_bfloat16* q_full;   // [B, H, 576]
  const float* q_sum;            // [B, H, kQSumParts] (INT8: the zero-point term)
  const void* cache;             // bf16 or int8 [num_pages, P, 576]
  const float* scale_zero;       // [num_pages, P, 2] (INT8) or [num_pages, P] (FP8)
  const int* block_table;        // [B, max_pages]
  const int* tile_start;
  const int* seg_base;
  const int* len;                // checked lengths
  float* partial_o;              // [NSEG, H, 512]
  float* partial_lse;            // [NSEG, H]
  int* status;
  int batch, heads, head_group, num_groups, page_size, max_pages, num_pages, num_splits;
  // multi-token decode: row v of a sequence is query token v / heads_w, at
  // position len - q_len + v / heads_w; it attends to positions up to its own
  int q_len, heads_w;
  float scale_log2;              // softmax_scale * log2(e)
  int inject_wait_timeout;       // test hook (mla_test_inject_wait_timeout): 16 bytes never delivered
};

__device__ inline void set_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

__device__ inline float bf2f(__nv_bfloat16 x) { return __bfloat162float(x); }

// Block-wide exclusive scan of `v` (one value per thread, blockDim.x <= 1024,
// multiple of 32).  Returns the exclusive prefix; *total gets the block sum.
__device__ inline int block_exclusive_scan(int v, int* smem32, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) smem32[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nwarps ? smem32[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    smem32[lane] = w;  // inclusive prefix of warp sums
  }
  __syncthreads();
  const int warp_prefix = warp ? smem32[warp - 1] : 0;
  *total = smem32[nwarps - 1];
  __syncthreads();
  return warp_prefix + x - v;
}

}  // namespace mla
