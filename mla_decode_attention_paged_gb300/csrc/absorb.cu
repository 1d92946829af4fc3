// absorb.cu -- query absorption and the decode work plan.
//
// Query absorption ("The Architecture of Memory", "The Weight Absorption
// Trick"; "Seven Ways LLMs Handle Attention", section 5): because
// q . (W^UK c) = (W^UK^T q) . c, each head's content query is mapped into
// latent space once per step, q_lat = W^UK_h^T q_nope (512 wide), and the
// attention kernel then scores the 576-wide cached rows directly with
// q_full = [q_lat | q_pe].
#include <cuda_fp16.h>

#include "params.cuh"

namespace mla {



// Block (0, 0) also computes the work plan before its share of the absorption.
__device__ void compute_plan(const AbsorbParams& p) {
  __shared__ int scan_tmp[32];
  __shared__ int carry;
  if (threadIdx.x == 0) {
    carry = 0;
    *p.status = MLA_OK;
  }
  __syncthreads();
  // pass 1: checked lengths, tiles per sequence, prefix sums -> tile_start
  for (int base = 0; base < p.batch; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int tiles = 0;
    if (b < p.batch) {
      int L = p.seq_lens[b];
      if (L < 0 || L > p.max_len) {
        set_status(p.status, MLA_ERR_DEVICE_BOUNDS);
        L = 0;
      }
      p.len_checked[b] = L;
      tiles = (L + kTile - 1) / kTile;
    }
    int total;
    const int ex = block_exclusive_scan(tiles, scan_tmp, &total);
    if (b < p.batch) p.tile_start[b] = carry + ex;
    __syncthreads();
    if (threadIdx.x == 0) carry += total;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    p.tile_start[p.batch] = carry;
    carry = 0;
  }
  __syncthreads();
  const long long W = p.tile_start[p.batch];
  const long long S = p.num_splits < W ? p.num_splits : (W > 0 ? W : 1);
  if (threadIdx.x == 0) p.status[1] = int(S);  // effective split count, read by the later kernels
  // pass 2: segments per sequence (partitions its tiles touch) -> seg_base
  for (int base = 0; base < p.batch; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int nseg = 0;
    if (b < p.batch) {
      const long long s = p.tile_start[b], e = p.tile_start[b + 1];
      if (e > s) nseg = int(part_of(e - 1, W, S) - part_of(s, W, S) + 1);
    }
    int total;
    const int ex = block_exclusive_scan(nseg, scan_tmp, &total);
    if (b < p.batch) p.seg_base[b] = carry + ex;
    __syncthreads();
    if (threadIdx.x == 0) carry += total;
    __syncthreads();
  }
  if (threadIdx.x == 0) p.seg_base[p.batch] = carry;
}

constexpr int kAbsM = 64;   // latent dims per block
constexpr int kAbsB = 32;   // sequences per pass

template <bool kF16>
__device__ __forceinline__ float round_out(float v, uint16_t* dst) {  // store as bf16/fp16, return the stored value
  if constexpr (kF16) {
    const __half r = __float2half_rn(v);
    *dst = __half_as_ushort(r);
    return __half2float(r);
  } else {
    const __nv_bfloat16 r = __float2bfloat16_rn(v);
    *dst = __bfloat16_as_ushort(r);
    return bf2f(r);
  }
}

// grid (H, 512 / 64), block 256.  Block (h, c) computes latent dims
// [64c, 64c + 64) of q_lat = W^UK_h^T q_nope for every sequence, with W^UK_h's
// columns staged in shared memory; thread (m, g) handles dim m for 8
// sequences per pass, fp32 accumulation over the 128 content dims.  Blocks
// (h, 0) also copy the RoPE part.  Part c of q_sum[b][h] is the sum of the
// rounded values the block wrote (part 0 includes the RoPE part).  INT8
// caches take q_full in fp16 (their tensor-core path runs on fp16 operands);
// bf16 caches in bf16.
template <bool kF16>
__global__ void __launch_bounds__(256) absorb_kernel(AbsorbParams p) {
  if (blockIdx.x == 0 && blockIdx.y == 0) {
    compute_plan(p);
    __syncthreads();
  }
  __shared__ __align__(16) __nv_bfloat16 ws[kNope][kAbsM];
  __shared__ __align__(16) float qs[kAbsB][kNope];
  __shared__ float red[kAbsB][2];
  const int h = blockIdx.x, c = blockIdx.y, tid = threadIdx.x, lane = tid & 31;
  const int m = tid & (kAbsM - 1), grp = tid >> 6;  // grp handles sequences 8 grp .. 8 grp + 7 of a pass
  for (int idx = tid; idx < kNope * kAbsM / 8; idx += blockDim.x) {
    const int k = idx >> 3, part = idx & 7;
    reinterpret_cast<uint4*>(&ws[k][0])[part] =
        *reinterpret_cast<const uint4*>(p.W_UK + (size_t(h) * kNope + k) * kLatent + c * kAbsM + part * 8);
  }
  uint16_t* qf = reinterpret_cast<uint16_t*>(p.q_full);
  for (int b0 = 0; b0 < p.batch; b0 += kAbsB) {
    const int nb = min(kAbsB, p.batch - b0);
    __syncthreads();  // ws loaded; qs and red free
    for (int idx = tid; idx < kAbsB * kNope / 8; idx += blockDim.x) {
      const int i = idx >> 4, part = idx & 15;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (i < nb) v = *reinterpret_cast<const uint4*>(p.q_nope + (size_t(b0 + i) * p.heads + h) * kNope + part * 8);
      const __nv_bfloat162* v2 = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(v2[e]);
        qs[i][part * 8 + 2 * e] = f.x;
        qs[i][part * 8 + 2 * e + 1] = f.y;
      }
    }
    __syncthreads();
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll 4
    for (int k = 0; k < kNope; k += 4) {
      const float w0 = bf2f(ws[k][m]), w1 = bf2f(ws[k + 1][m]), w2 = bf2f(ws[k + 2][m]), w3 = bf2f(ws[k + 3][m]);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 q = *reinterpret_cast<const float4*>(&qs[8 * grp + i][k]);  // same address across the warp
        acc[i] = fmaf(w3, q.w, fmaf(w2, q.z, fmaf(w1, q.y, fmaf(w0, q.x, acc[i]))));
      }
    }
    // round, store and sum this block's part of each sequence's q_full row
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int bi = 8 * grp + i;
      float r = 0.f;
      if (bi < nb) r = round_out<kF16>(acc[i], qf + (size_t(b0 + bi) * p.heads + h) * kRow + c * kAbsM + m);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
      if (lane == 0) red[bi][(tid >> 5) & 1] = r;
    }
    __syncthreads();
    // RoPE part (blocks c == 0): eight threads per sequence, eight values each
    const int bi = tid >> 3, r8 = tid & 7;
    float rope = 0.f;
    if (c == 0) {
      if (bi < nb) {
        const size_t row = size_t(b0 + bi) * p.heads + h;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int d = r8 * 8 + e;
          rope += round_out<kF16>(bf2f(p.q_pe[row * kRope + d]), qf + row * kRow + kLatent + d);
        }
      }
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) rope += __shfl_xor_sync(0xffffffffu, rope, o);
    }
    if (r8 == 0 && bi < nb)
      p.q_sum[(size_t(b0 + bi) * p.heads + h) * kQSumParts + c] = (red[bi][0] + red[bi][1]) + rope;
  }
}

cudaError_t launch_absorb(const AbsorbParams& p, bool fp16_out, cudaStream_t stream) {
  dim3 grid(p.heads, kLatent / kAbsM);
  static_assert(kLatent / kAbsM == kQSumParts, "one q_sum part per block of latent dims");
  if (fp16_out) absorb_kernel<true><<<grid, 256, 0, stream>>>(p);
  else absorb_kernel<false><<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mla
