// combine.cu -- log-sum-exp merge of split-KV partials ("The Architecture of
// Memory", "Flash-Decoding and FlashInfer": each chunk yields a partial
// result and the partials are merged by a log-sum-exp reduction) and the
// value up-projection that the absorbed form applies last ("The Weight
// Absorption Trick"; "Seven Ways LLMs Handle Attention", section 5: the value
// expansion is absorbed into the output side): out_h = W^UV_h o_lat_h.
#include "params.cuh"

namespace mla {


constexpr int kCombB = 8;     // sequences per block
constexpr int kCombJ = 64;    // output dims per block (of 128)

constexpr int kMergeWarps = 16;  // at most

// grid (H, B), block 32 nw (nw <= 16 warps, chosen from the average number
// of segments per sequence): the LSE merge of the segments of sequence b,
// head h.  Warp w takes segments w, w + nw, ...; lane l accumulates latent
// dims [16 l, 16 l + 16); the warps' sums are added in warp order (the result
// does not depend on timing).
__global__ void __launch_bounds__(kMergeWarps * 32) merge_kernel(CombineUVParams p) {
  extern __shared__ __align__(16) float part_raw[];  // [nw][kLatent]
  __shared__ float red[kMergeWarps];
  const int nw = blockDim.x >> 5;
  __shared__ float s_mx, s_z;
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int s0 = p.seg_base[b], s1 = p.seg_base[b + 1];
  // lse of the merged result: max, then sum of exp(lse_s - max)
  float mx = -INFINITY;
  for (int s = s0 + tid; s < s1; s += blockDim.x) mx = fmaxf(mx, p.partial_lse[size_t(s) * p.heads + h]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  if (tid == 0) {
    float v = red[0];
    for (int k = 1; k < nw; ++k) v = fmaxf(v, red[k]);
    s_mx = v;
  }
  __syncthreads();
  mx = s_mx;
  float z = 0.f;
  if (mx != -INFINITY)
    for (int s = s0 + tid; s < s1; s += blockDim.x) z += expf(p.partial_lse[size_t(s) * p.heads + h] - mx);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  __syncthreads();
  if (lane == 0) red[warp] = z;
  __syncthreads();
  if (tid == 0) {
    float v = 0.f;
    for (int k = 0; k < nw; ++k) v += red[k];
    s_z = v;
    if (p.lse_out) p.lse_out[size_t(b) * p.heads + h] = mx != -INFINITY ? mx + logf(v) : -INFINITY;
  }
  __syncthreads();
  const float inv_z = mx != -INFINITY ? 1.f / s_z : 0.f;
  float4 acc[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (mx != -INFINITY)
    for (int s = s0 + warp; s < s1; s += nw) {
      const float w = expf(p.partial_lse[size_t(s) * p.heads + h] - mx) * inv_z;
      const float4* src = reinterpret_cast<const float4*>(p.partial_o + (size_t(s) * p.heads + h) * kLatent) + 4 * lane;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 v = src[q];
        acc[q].x = fmaf(w, v.x, acc[q].x);
        acc[q].y = fmaf(w, v.y, acc[q].y);
        acc[q].z = fmaf(w, v.z, acc[q].z);
        acc[q].w = fmaf(w, v.w, acc[q].w);
      }
    }
  float* dst = p.o_lat + (size_t(b) * p.heads + h) * kLatent;
  if (nw == 1) {
#pragma unroll
    for (int q = 0; q < 4; ++q) reinterpret_cast<float4*>(dst)[4 * lane + q] = acc[q];
    return;
  }
  float4* mine = reinterpret_cast<float4*>(part_raw + warp * kLatent) + 4 * lane;
#pragma unroll
  for (int q = 0; q < 4; ++q) mine[q] = acc[q];
  __syncthreads();
  for (int d = tid; d < kLatent; d += blockDim.x) {
    float v = part_raw[d];
    for (int k = 1; k < nw; ++k) v += part_raw[k * kLatent + d];
    dst[d] = v;
  }
}

// grid (H, ceil(B / 8), 128 / 64), block 256: out[b][h][j] = W^UV_h[j] . o_lat[b][h]
// for 8 sequences and output rows [64 z, 64 z + 64).
__global__ void __launch_bounds__(256) combine_uv_kernel(CombineUVParams p) {
  __shared__ __align__(16) float o_lat[kCombB][kLatent];
  const int h = blockIdx.x, b0 = blockIdx.y * kCombB, j0 = blockIdx.z * kCombJ;
  const int nb = min(kCombB, p.batch - b0);
  const int tid = threadIdx.x;
  for (int idx = tid; idx < kCombB * kLatent / 4; idx += blockDim.x) {
    const int i = idx / (kLatent / 4), q = idx % (kLatent / 4);
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (i < nb) v = reinterpret_cast<const float4*>(p.o_lat + (size_t(b0 + i) * p.heads + h) * kLatent)[q];
    reinterpret_cast<float4*>(o_lat[i])[q] = v;
  }
  __syncthreads();

  // out[b][h][j] = sum_m W_UV[h][j][m] * o_lat[b][m]: warp w takes rows j0 + w, j0 + w + 8, ...;
  // lane l covers dims 128 r + 4 l + (0..3), r < 4 (coalesced rows, conflict-free shared reads)
  const int warp = tid >> 5, lane = tid & 31;
  for (int jj = warp; jj < kCombJ; jj += 8) {
    const int j = j0 + jj;
    const uint2* wrow = reinterpret_cast<const uint2*>(p.W_UV + (size_t(h) * kVDim + j) * kLatent);
    float wf[16];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const uint2 wv = wrow[32 * r + lane];
      const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wv.x));
      const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wv.y));
      wf[4 * r] = x.x;
      wf[4 * r + 1] = x.y;
      wf[4 * r + 2] = y.x;
      wf[4 * r + 3] = y.y;
    }
    float acc[kCombB];
#pragma unroll
    for (int i = 0; i < kCombB; ++i) {
      float a = 0.f;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float4 o = reinterpret_cast<const float4*>(o_lat[i])[32 * r + lane];
        a = fmaf(wf[4 * r], o.x, fmaf(wf[4 * r + 1], o.y, fmaf(wf[4 * r + 2], o.z, fmaf(wf[4 * r + 3], o.w, a))));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
      acc[i] = a;
    }
    float mine = acc[0];
#pragma unroll
    for (int i = 1; i < kCombB; ++i)
      if (lane == i) mine = acc[i];
    if (lane < nb) p.out[(size_t(b0 + lane) * p.heads + h) * kVDim + j] = __float2bfloat16_rn(mine);
  }
}

cudaError_t launch_combine_uv(const CombineUVParams& p, cudaStream_t stream) {
  // about two segments per warp
  int nw = 1;
  while (nw < kMergeWarps && 2 * nw * p.batch < p.max_segments) nw *= 2;
  merge_kernel<<<dim3(p.heads, p.batch), nw * 32, nw > 1 ? nw * kLatent * sizeof(float) : 0, stream>>>(p);
  dim3 grid(p.heads, (p.batch + kCombB - 1) / kCombB, kVDim / kCombJ);
  combine_uv_kernel<<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

// ----- standalone combine (mla_combine) ---------------------------------------

// grid (H, B), block 128
__global__ void __launch_bounds__(128) combine_kernel(CombineParams p) {
  const int h = blockIdx.x, b = blockIdx.y;
  float mx = -INFINITY;
  for (int s = 0; s < p.splits; ++s) mx = fmaxf(mx, p.partial_lse[(size_t(b) * p.splits + s) * p.heads + h]);
  float z = 0.f;
  if (mx != -INFINITY)
    for (int s = 0; s < p.splits; ++s) z += expf(p.partial_lse[(size_t(b) * p.splits + s) * p.heads + h] - mx);
  const float inv_z = mx != -INFINITY ? 1.f / z : 0.f;
  for (int d = threadIdx.x; d < p.dim; d += blockDim.x) {
    float acc = 0.f;
    if (mx != -INFINITY)
      for (int s = 0; s < p.splits; ++s) {
        const size_t bs = size_t(b) * p.splits + s;
        const float w = expf(p.partial_lse[bs * p.heads + h] - mx);
        acc = fmaf(w, p.partial_o[(bs * p.heads + h) * p.dim + d], acc);
      }
    p.o_lat[(size_t(b) * p.heads + h) * p.dim + d] = acc * inv_z;
  }
  if (threadIdx.x == 0 && p.lse_out)
    p.lse_out[size_t(b) * p.heads + h] = mx != -INFINITY ? mx + logf(z) : -INFINITY;
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream) {
  dim3 grid(p.heads, p.batch);
  combine_kernel<<<grid, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mla
