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
constexpr int kSegChunk = 256;

// grid (H, ceil(B / 8), 128 / 64), block 256.  Phase 1 merges the segments of
// 8 sequences of head h into shared memory (weights exp(lse_s - lse) computed
// once per segment); phase 2 multiplies them by rows [64z, 64z + 64) of W^UV_h.
__global__ void __launch_bounds__(256) combine_uv_kernel(CombineUVParams p) {
  __shared__ float o_lat[kCombB][kLatent];
  __shared__ float wts[kSegChunk];
  __shared__ float red[8];
  __shared__ float s_mx, s_inv_z;
  const int h = blockIdx.x, b0 = blockIdx.y * kCombB, j0 = blockIdx.z * kCombJ;
  const int nb = min(kCombB, p.batch - b0);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  for (int i = 0; i < kCombB; ++i) {
    if (i >= nb) {
      for (int m = tid; m < kLatent; m += blockDim.x) o_lat[i][m] = 0.f;
      continue;
    }
    const int b = b0 + i;
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
      for (int k = 1; k < 8; ++k) v = fmaxf(v, red[k]);
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
      for (int k = 0; k < 8; ++k) v += red[k];
      s_inv_z = mx != -INFINITY ? 1.f / v : 0.f;
      if (p.lse_out && blockIdx.z == 0)
        p.lse_out[size_t(b) * p.heads + h] = mx != -INFINITY ? mx + logf(v) : -INFINITY;
    }
    __syncthreads();
    const float inv_z = s_inv_z;
    float acc0 = 0.f, acc1 = 0.f;
    if (mx != -INFINITY) {
      for (int c0 = s0; c0 < s1; c0 += kSegChunk) {
        const int n = min(kSegChunk, s1 - c0);
        __syncthreads();
        for (int k = tid; k < n; k += blockDim.x) wts[k] = expf(p.partial_lse[size_t(c0 + k) * p.heads + h] - mx) * inv_z;
        __syncthreads();
        for (int k = 0; k < n; ++k) {
          const float* src = p.partial_o + (size_t(c0 + k) * p.heads + h) * kLatent;
          acc0 = fmaf(wts[k], src[tid], acc0);
          acc1 = fmaf(wts[k], src[tid + 256], acc1);
        }
      }
    }
    o_lat[i][tid] = acc0;
    o_lat[i][tid + 256] = acc1;
    __syncthreads();
  }

  // out[b][h][j] = sum_m W_UV[h][j][m] * o_lat[b][m]; thread -> (j, pair of sequences)
  const int j = j0 + (tid & 63), bp = tid >> 6;
  const uint4* wrow = reinterpret_cast<const uint4*>(p.W_UV + (size_t(h) * kVDim + j) * kLatent);
  float a0 = 0.f, a1 = 0.f;
#pragma unroll 4
  for (int k8 = 0; k8 < kLatent / 8; ++k8) {
    const uint4 wv = wrow[k8];
    const __nv_bfloat162* w2 = reinterpret_cast<const __nv_bfloat162*>(&wv);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 wf = __bfloat1622float2(w2[e]);
      const int m = 8 * k8 + 2 * e;
      a0 = fmaf(wf.x, o_lat[2 * bp][m], fmaf(wf.y, o_lat[2 * bp][m + 1], a0));
      a1 = fmaf(wf.x, o_lat[2 * bp + 1][m], fmaf(wf.y, o_lat[2 * bp + 1][m + 1], a1));
    }
  }
  if (2 * bp < nb) p.out[(size_t(b0 + 2 * bp) * p.heads + h) * kVDim + j] = __float2bfloat16_rn(a0);
  if (2 * bp + 1 < nb) p.out[(size_t(b0 + 2 * bp + 1) * p.heads + h) * kVDim + j] = __float2bfloat16_rn(a1);
}

cudaError_t launch_combine_uv(const CombineUVParams& p, cudaStream_t stream) {
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
