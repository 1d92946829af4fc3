// decode_simt.cu -- bring-up split-KV attention on CUDA cores.  Same work
// plan and partial-result format as the tensor-core kernel; used to validate
// the plan, combine and projection steps independently of tcgen05.
#include "params.cuh"

namespace mla {

template <int HC, bool kInt8>
__global__ void __launch_bounds__(256) decode_simt_kernel(DecodeParams p) {
  extern __shared__ float smem[];
  float* qs = smem;                            // [HC][576] q_full of this segment
  float* sc = qs + HC * kRow;                  // [128][HC + 1] scores, then weights
  float* m_run = sc + kTile * (HC + 1);        // [HC]
  float* l_run = m_run + HC;                   // [HC]
  float* alpha_s = l_run + HC;                 // [HC]
  int* rowidx = reinterpret_cast<int*>(alpha_s + HC);  // [128] physical row per token, -1 = none
  float* rowscale = reinterpret_cast<float*>(rowidx + kTile);  // [128][2] (INT8)

  const int G = p.num_groups, g = blockIdx.x % G, cp = blockIdx.x / G, Cp = gridDim.x / G;
  const long long S = p.status[1];  // effective split count from the plan
  const long long pa = (cp * S) / Cp, pb = ((cp + 1) * S) / Cp;
  TileWalker walk;
  walk.init(p.tile_start, p.seg_base, p.len, p.batch, int(S), pa, pb);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h0 = g * HC;
  float acc_o[HC][2];
  TileInfo t;
  while (walk.next(t)) {
    if (t.first) {
      __syncthreads();
      for (int i = tid; i < HC * kRow; i += blockDim.x) {
        const int h = i / kRow, d = i % kRow;
        qs[i] = bf2f(p.q_full[(size_t(t.b) * p.heads + h0 + h) * kRow + d]);
      }
      if (tid < HC) {
        m_run[tid] = -INFINITY;
        l_run[tid] = 0.f;
      }
#pragma unroll
      for (int h = 0; h < HC; ++h) acc_o[h][0] = acc_o[h][1] = 0.f;
    }
    if (tid < kTile) {
      int ri = -1;
      if (tid < t.valid) {
        const int tok = t.tile * kTile + tid;
        const int page = p.block_table[size_t(t.b) * p.max_pages + tok / p.page_size];
        if (page >= 0 && page < p.num_pages) ri = page * p.page_size + tok % p.page_size;
        else set_status(p.status, MLA_ERR_DEVICE_BOUNDS);
      }
      rowidx[tid] = ri;
      if (kInt8 && ri >= 0) {
        rowscale[2 * tid] = p.scale_zero[size_t(ri) * 2];
        rowscale[2 * tid + 1] = p.scale_zero[size_t(ri) * 2 + 1];
      }
    }
    __syncthreads();
    // scores: token tt = tid & 127 over the dims of half (tid >> 7)
    {
      const int tt = tid & 127, half = tid >> 7;
      float acc[HC];
#pragma unroll
      for (int h = 0; h < HC; ++h) acc[h] = 0.f;
      const int ri = rowidx[tt];
      if (ri >= 0) {
        if constexpr (!kInt8) {
          const uint4* r = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.cache) + size_t(ri) * kRow + half * (kRow / 2));
          for (int j = 0; j < kRow / 2 / 8; ++j) {
            uint4 v = r[j];
            const __nv_bfloat162* v2 = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float x0 = __low2float(v2[e]), x1 = __high2float(v2[e]);
              const int d = half * (kRow / 2) + j * 8 + 2 * e;
#pragma unroll
              for (int h = 0; h < HC; ++h) acc[h] = fmaf(qs[h * kRow + d + 1], x1, fmaf(qs[h * kRow + d], x0, acc[h]));
            }
          }
        } else {
          const float s = rowscale[2 * tt], z = rowscale[2 * tt + 1];
          const int8_t* r = static_cast<const int8_t*>(p.cache) + size_t(ri) * kRow + half * (kRow / 2);
          for (int j = 0; j < kRow / 2; ++j) {
            const float x = s * (float(r[j]) - z);
            const int d = half * (kRow / 2) + j;
#pragma unroll
            for (int h = 0; h < HC; ++h) acc[h] = fmaf(qs[h * kRow + d], x, acc[h]);
          }
        }
      }
      if (half == 1)
#pragma unroll
        for (int h = 0; h < HC; ++h) sc[tt * (HC + 1) + h] = acc[h];
      __syncthreads();
      if (half == 0)
#pragma unroll
        for (int h = 0; h < HC; ++h)
          sc[tt * (HC + 1) + h] = ri >= 0 ? (sc[tt * (HC + 1) + h] + acc[h]) * p.scale_log2 : -INFINITY;
      __syncthreads();
    }
    // online softmax per head (base 2)
    for (int h = warp; h < HC; h += 8) {
      float x[4], mt = -INFINITY;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        x[k] = sc[(lane + 32 * k) * (HC + 1) + h];
        mt = fmaxf(mt, x[k]);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
      const float m_old = m_run[h];
      const float m_new = fmaxf(m_old, mt);
      const float alpha = exp2f(m_old - m_new);
      float sum = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float pr = exp2f(x[k] - m_new);
        sc[(lane + 32 * k) * (HC + 1) + h] = pr;
        sum += pr;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      __syncwarp();
      if (lane == 0) {
        l_run[h] = l_run[h] * alpha + sum;
        m_run[h] = m_new;
        alpha_s[h] = alpha;
      }
    }
    __syncthreads();
    // weighted latent sum: thread owns latent dims tid and tid + 256
#pragma unroll
    for (int h = 0; h < HC; ++h) {
      acc_o[h][0] *= alpha_s[h];
      acc_o[h][1] *= alpha_s[h];
    }
    for (int tt = 0; tt < t.valid; ++tt) {
      const int ri = rowidx[tt];
      if (ri < 0) continue;
      float c0, c1;
      if constexpr (!kInt8) {
        const __nv_bfloat16* r = static_cast<const __nv_bfloat16*>(p.cache) + size_t(ri) * kRow;
        c0 = bf2f(r[tid]);
        c1 = bf2f(r[tid + 256]);
      } else {
        const int8_t* r = static_cast<const int8_t*>(p.cache) + size_t(ri) * kRow;
        const float s = rowscale[2 * tt], z = rowscale[2 * tt + 1];
        c0 = s * (float(r[tid]) - z);
        c1 = s * (float(r[tid + 256]) - z);
      }
#pragma unroll
      for (int h = 0; h < HC; ++h) {
        const float w = sc[tt * (HC + 1) + h];
        acc_o[h][0] = fmaf(w, c0, acc_o[h][0]);
        acc_o[h][1] = fmaf(w, c1, acc_o[h][1]);
      }
    }
    __syncthreads();
    if (t.last) {
#pragma unroll
      for (int h = 0; h < HC; ++h) {
        const float inv = 1.f / l_run[h];
        float* dst = p.partial_o + (size_t(t.seg) * p.heads + h0 + h) * kLatent;
        dst[tid] = acc_o[h][0] * inv;
        dst[tid + 256] = acc_o[h][1] * inv;
      }
      if (tid < HC) p.partial_lse[size_t(t.seg) * p.heads + h0 + tid] = (m_run[tid] + log2f(l_run[tid])) * kLn2;
    }
  }
}

size_t simt_smem_bytes(int hc) {
  return (size_t(hc) * kRow + kTile * (hc + 1) + 3 * hc) * 4 + kTile * 4 + kTile * 8;
}

template <int HC, bool kInt8>
static cudaError_t launch_simt_t(const DecodeParams& p, int grid, cudaStream_t stream) {
  const size_t smem = simt_smem_bytes(HC);
  cudaError_t e = cudaFuncSetAttribute(decode_simt_kernel<HC, kInt8>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  decode_simt_kernel<HC, kInt8><<<grid, 256, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_decode_simt(const DecodeParams& p, int hc, bool int8, int grid, cudaStream_t stream) {
  if (hc == 16) return int8 ? launch_simt_t<16, true>(p, grid, stream) : launch_simt_t<16, false>(p, grid, stream);
  return int8 ? launch_simt_t<32, true>(p, grid, stream) : launch_simt_t<32, false>(p, grid, stream);
}

}  // namespace mla
