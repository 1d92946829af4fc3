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


constexpr int kAbsorbB = 8;  // sequences per block

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

// grid (H, ceil(B / 8)), block 512: thread m computes latent dim m of q_lat
// for 8 sequences of head h, fp32 accumulation over the 128 content dims.
// INT8 caches take q_full in fp16 (their tensor-core path runs on fp16
// operands); bf16 caches in bf16.
template <bool kF16>
__global__ void __launch_bounds__(512) absorb_kernel(AbsorbParams p) {
  if (blockIdx.x == 0 && blockIdx.y == 0) {
    compute_plan(p);
    __syncthreads();
  }
  __shared__ float4 qs[kNope][kAbsorbB / 4];  // q_nope[b0 + i][h][k] at qs[k][i / 4].{x,y,z,w}
  __shared__ float red[kAbsorbB][16];
  const int h = blockIdx.x, b0 = blockIdx.y * kAbsorbB;
  const int nb = min(kAbsorbB, p.batch - b0);
  float* qsf = reinterpret_cast<float*>(qs);
  for (int idx = threadIdx.x; idx < kAbsorbB * kNope; idx += blockDim.x) {
    const int i = idx / kNope, k = idx % kNope;
    float v = 0.f;
    if (i < nb) v = bf2f(p.q_nope[(size_t(b0 + i) * p.heads + h) * kNope + k]);
    qsf[k * kAbsorbB + i] = v;
  }
  __syncthreads();
  const int m = threadIdx.x;
  float acc[kAbsorbB];
#pragma unroll
  for (int i = 0; i < kAbsorbB; ++i) acc[i] = 0.f;
  const __nv_bfloat16* w = p.W_UK + size_t(h) * kNope * kLatent + m;
#pragma unroll 8
  for (int k = 0; k < kNope; ++k) {
    const float wk = bf2f(w[size_t(k) * kLatent]);
#pragma unroll
    for (int i4 = 0; i4 < kAbsorbB / 4; ++i4) {
      const float4 q = qs[k][i4];
      acc[4 * i4 + 0] = fmaf(wk, q.x, acc[4 * i4 + 0]);
      acc[4 * i4 + 1] = fmaf(wk, q.y, acc[4 * i4 + 1]);
      acc[4 * i4 + 2] = fmaf(wk, q.z, acc[4 * i4 + 2]);
      acc[4 * i4 + 3] = fmaf(wk, q.w, acc[4 * i4 + 3]);
    }
  }
  // write q_full[b][h][0:512] (and the RoPE part) and the sum of the rounded values
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint16_t* qf = reinterpret_cast<uint16_t*>(p.q_full);
#pragma unroll
  for (int i = 0; i < kAbsorbB; ++i) {
    float r = 0.f;
    if (i < nb) {
      const size_t row = (size_t(b0 + i) * p.heads + h) * kRow;
      if constexpr (kF16) {
        const __half v = __float2half_rn(acc[i]);
        qf[row + m] = __half_as_ushort(v);
        r = __half2float(v);
      } else {
        const __nv_bfloat16 v = __float2bfloat16_rn(acc[i]);
        qf[row + m] = __bfloat16_as_ushort(v);
        r = bf2f(v);
      }
      if (threadIdx.x < kRope) {
        const float pe = bf2f(p.q_pe[(size_t(b0 + i) * p.heads + h) * kRope + threadIdx.x]);
        if constexpr (kF16) {
          const __half v = __float2half_rn(pe);
          qf[row + kLatent + threadIdx.x] = __half_as_ushort(v);
          r += __half2float(v);
        } else {
          qf[row + kLatent + threadIdx.x] = __bfloat16_as_ushort(__float2bfloat16_rn(pe));
          r += pe;
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
    if (lane == 0) red[i][warp] = r;
  }
  __syncthreads();
  if (threadIdx.x < nb) {
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) s += red[threadIdx.x][j];
    p.q_sum[size_t(b0 + threadIdx.x) * p.heads + h] = s;
  }
}

cudaError_t launch_absorb(const AbsorbParams& p, bool fp16_out, cudaStream_t stream) {
  dim3 grid(p.heads, (p.batch + kAbsorbB - 1) / kAbsorbB);
  if (fp16_out) absorb_kernel<true><<<grid, 512, 0, stream>>>(p);
  else absorb_kernel<false><<<grid, 512, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mla
