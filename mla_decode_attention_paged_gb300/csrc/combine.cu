// combine.cu -- log-sum-exp merge of split-KV partials ("The Architecture of
// Memory", "Flash-Decoding and FlashInfer": each chunk yields a partial
// result and the partials are merged by a log-sum-exp reduction) and the
// value up-projection that the absorbed form applies last ("The Weight
// Absorption Trick"; "Seven Ways LLMs Handle Attention", section 5: the value
// expansion is absorbed into the output side): out_h = W^UV_h o_lat_h.
#include "params.cuh"

namespace mla {


constexpr int kCombB = 32;   // sequences per block
constexpr int kCombMK = 64;  // latent dims per W^UV tile

// grid (H, ceil(B / 32)), block 256.  Phase 1 merges the partials of 32
// sequences of head h into shared memory; phase 2 multiplies them by W^UV_h.
__global__ void __launch_bounds__(256) combine_uv_kernel(CombineUVParams p) {
  extern __shared__ float smem[];
  float* o_lat = smem;                          // [32][512]
  float* w_tile = smem + kCombB * kLatent;      // [128][kCombMK + 1]
  const int h = blockIdx.x, b0 = blockIdx.y * kCombB;
  const int nb = min(kCombB, p.batch - b0);

  for (int i = 0; i < kCombB; ++i) {
    float* row = o_lat + i * kLatent;
    if (i >= nb) {
      for (int m = threadIdx.x; m < kLatent; m += blockDim.x) row[m] = 0.f;
      continue;
    }
    const int b = b0 + i;
    const int s0 = p.seg_base[b], s1 = p.seg_base[b + 1];
    float mx = -INFINITY;
    for (int s = s0; s < s1; ++s) mx = fmaxf(mx, p.partial_lse[size_t(s) * p.heads + h]);
    float z = 0.f;
    if (mx != -INFINITY)
      for (int s = s0; s < s1; ++s) z += expf(p.partial_lse[size_t(s) * p.heads + h] - mx);
    const float inv_z = mx != -INFINITY ? 1.f / z : 0.f;
    for (int m = threadIdx.x; m < kLatent; m += blockDim.x) {
      float acc = 0.f;
      if (mx != -INFINITY)
        for (int s = s0; s < s1; ++s) {
          const float w = expf(p.partial_lse[size_t(s) * p.heads + h] - mx);
          acc = fmaf(w, p.partial_o[(size_t(s) * p.heads + h) * kLatent + m], acc);
        }
      row[m] = acc * inv_z;
    }
    if (threadIdx.x == 0 && p.lse_out)
      p.lse_out[size_t(b) * p.heads + h] = mx != -INFINITY ? mx + logf(z) : -INFINITY;
  }

  // out[b][h][j] = sum_m W_UV[h][j][m] * o_lat[b][m]; thread -> (j, half of the 32 sequences)
  const int j = threadIdx.x & 127, half = threadIdx.x >> 7;
  float acc[kCombB / 2];
#pragma unroll
  for (int i = 0; i < kCombB / 2; ++i) acc[i] = 0.f;
  const __nv_bfloat16* W = p.W_UV + size_t(h) * kVDim * kLatent;
  for (int m0 = 0; m0 < kLatent; m0 += kCombMK) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < kVDim * kCombMK; idx += blockDim.x) {
      const int jj = idx / kCombMK, mm = idx % kCombMK;
      w_tile[jj * (kCombMK + 1) + mm] = bf2f(W[size_t(jj) * kLatent + m0 + mm]);
    }
    __syncthreads();
#pragma unroll 4
    for (int mm = 0; mm < kCombMK; ++mm) {
      const float w = w_tile[j * (kCombMK + 1) + mm];
#pragma unroll
      for (int i = 0; i < kCombB / 2; ++i)
        acc[i] = fmaf(w, o_lat[(half * (kCombB / 2) + i) * kLatent + m0 + mm], acc[i]);
    }
  }
#pragma unroll
  for (int i = 0; i < kCombB / 2; ++i) {
    const int bi = half * (kCombB / 2) + i;
    if (bi < nb) p.out[(size_t(b0 + bi) * p.heads + h) * kVDim + j] = __float2bfloat16_rn(acc[i]);
  }
}

cudaError_t launch_combine_uv(const CombineUVParams& p, cudaStream_t stream) {
  const size_t smem = (kCombB * kLatent + kVDim * (kCombMK + 1)) * sizeof(float);
  static bool attr_set[128] = {};  // per device; a repeated set is harmless
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 128 || !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(combine_uv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 128) attr_set[dev] = true;
  }
  dim3 grid(p.heads, (p.batch + kCombB - 1) / kCombB);
  combine_uv_kernel<<<grid, 256, smem, stream>>>(p);
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
