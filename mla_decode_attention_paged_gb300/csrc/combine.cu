// combine.cu -- log-sum-exp merge of split-KV partials ("The Architecture of
// Memory", "Flash-Decoding and FlashInfer": each chunk yields a partial
// result and the partials are merged by a log-sum-exp reduction) and the
// value up-projection that the absorbed form applies last ("The Weight
// Absorption Trick"; "Seven Ways LLMs Handle Attention", section 5: the value
// expansion is absorbed into the output side): out_h = W^UV_h o_lat_h.
#include <atomic>
#include "blackwell_ptx.cuh"
#include "decode_common.cuh"
#include "params.cuh"

namespace mla {

using namespace ptx;

// ---------------------------------------------------------------------------
// Merge and up-projection in one kernel.  A CTA takes one weight head h and
// NB query columns -- a column c = b * q_len + t is query token t of
// sequence b, whose row t * heads_w + h uses head h's weights:
//   1. its 16 warps merge each column's segments (the partial outputs of its
//      sequence's split-KV ranges) with log-sum-exp weights into o_lat (fp32), and
//      store it in shared memory as two bf16 rows, hi = bf16(o) and
//      lo = bf16(o - hi), which carry o to about 2^-16 relative;
//   2. one thread issues D [128 x 2 NB] = W^UV_h [128 x 512] * [hi | lo]^T on
//      the tensor cores (32 K = 16 MMAs, fp32 accumulation in TMEM; the hi
//      rows are D's first NB columns, the lo rows its last NB), with W^UV_h
//      (exact in bf16) brought in by TMA while the warps merge;
//   3. one thread per output dim j stores out[c][h][j] = D[j][c] + D[j][NB + c]
//      (bf16) for the tile's columns.
// Both operands are K-major with 128-byte swizzle, in blocks of 64 latent
// dims: W^UV_h block kb = rows j x dims [64 kb, 64 kb + 64) (16 KB), and the
// [hi | lo] block kb = 2 NB rows x the same dims.
constexpr int kUVWarps = 16;
constexpr int kUVThreads = 32 * kUVWarps;
constexpr int kUVBatch = 4;                  // segment rows a warp loads at once
constexpr uint32_t kUVWBlock = kVDim * 128;  // 16 KB
constexpr uint32_t kUVWBytes = 8 * kUVWBlock;
constexpr uint64_t kUVWaitNs = 2000000000ull;

template <int NB>
struct UVCfg {
  static_assert(NB == 8 || NB == 16 || NB == 32, "MMA N = 2 NB in 16 .. 64");
  static constexpr uint32_t kBBlock = 2 * NB * 128;
  static constexpr uint32_t kOffB = kUVWBytes;
  static constexpr uint32_t kOffX = kOffB + 8 * kBBlock;  // [kUVWarps][512] fp32 cross-warp sums
  static constexpr uint32_t kOffSeg = kOffX + kUVWarps * kLatent * 4;  // per column: first segment, row; NB + 1 ends
  static constexpr uint32_t kOffMisc = kOffSeg + 512;
  static constexpr uint32_t kSmem = kOffMisc + 64 + 1024;
  static constexpr uint32_t kTmemCols = 2 * NB < 32 ? 32 : 2 * NB;
  static_assert(kSmem <= 232448, "dynamic shared memory of one CTA");
};

// bf16 hi/lo split of 8 consecutive values of sequence row r, latent dims
// [d, d + 8) (d a multiple of 8), into rows r (hi) and NB + r (lo) of the
// swizzled B operand
template <int NB>
__device__ __forceinline__ void store_planes(uint8_t* bsm, int r, int d, const float* v) {
  uint32_t ph[4], pl[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const __nv_bfloat16 h0 = __float2bfloat16_rn(v[2 * e]), h1 = __float2bfloat16_rn(v[2 * e + 1]);
    const __nv_bfloat16 l0 = __float2bfloat16_rn(v[2 * e] - __bfloat162float(h0));
    const __nv_bfloat16 l1 = __float2bfloat16_rn(v[2 * e + 1] - __bfloat162float(h1));
    ph[e] = uint32_t(__bfloat16_as_ushort(h0)) | (uint32_t(__bfloat16_as_ushort(h1)) << 16);
    pl[e] = uint32_t(__bfloat16_as_ushort(l0)) | (uint32_t(__bfloat16_as_ushort(l1)) << 16);
  }
  // rows r and NB + r share r % 8, hence the 16-byte slot
  const uint32_t off = (d >> 6) * UVCfg<NB>::kBBlock + r * 128 + ((((d >> 3) & 7) ^ (r & 7)) << 4);
  *reinterpret_cast<uint4*>(bsm + off) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
  *reinterpret_cast<uint4*>(bsm + off + NB * 128) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
}

template <int NB>
__global__ void __launch_bounds__(kUVThreads, 1)
    merge_uv_kernel(const __grid_constant__ CUtensorMap tmap_wuv, CombineUVParams p) {
  using C = UVCfg<NB>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* w_full = reinterpret_cast<uint64_t*>(smem + C::kOffMisc);
  uint64_t* mma_done = w_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc + 16);
  int* abort_flag = reinterpret_cast<int*>(smem + C::kOffMisc + 20);
  uint8_t* bsm = smem + C::kOffB;
  float* xs = reinterpret_cast<float*>(smem + C::kOffX);
  int* seg_lo = reinterpret_cast<int*>(smem + C::kOffSeg);  // [NB] first segment of the column's sequence
  int* seg_hi = seg_lo + NB;                                  // [NB] its end
  int* row_of = seg_hi + NB;                                  // [NB] the column's row within its sequence
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cols = p.batch * p.q_len;
  const int per_head = (cols + NB - 1) / NB;
  const int h = blockIdx.x / per_head, b0 = (blockIdx.x % per_head) * NB, nb = min(NB, cols - b0);
  if (tid == 0) {
    mbar_init(w_full, 1);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmap_wuv);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  // This grid starts only after every CTA of the attention kernel has passed
  // its own wait, i.e. after the absorption kernel (and, through its wait,
  // everything before the call) completed.  So seg_base (written by the
  // absorption kernel) and W^UV (an input no kernel of the call writes) can
  // be read before the wait below, which covers the attention kernel's
  // partial results: W^UV's copy then runs under the attention kernel's tail.
  if (tid == 0) {
    mbar_arrive_expect_tx(w_full, kUVWBytes);
#pragma unroll
    for (int kb = 0; kb < 8; ++kb)
      tma_load_2d(smem + kb * kUVWBlock, &tmap_wuv, 64 * kb, h * kVDim, w_full);
  }
  if (tid < nb) {
    const int b = (b0 + tid) / p.q_len;
    seg_lo[tid] = p.seg_base[b];
    seg_hi[tid] = p.seg_base[b + 1];
    row_of[tid] = ((b0 + tid) % p.q_len) * p.heads_w + h;
  }
  griddep_wait();
  griddep_launch_dependents();
  __syncthreads();

  // ---- 1. merge.  wps warps per column (about kUVBatch segments each, as
  // far as the tile's columns still fit in one round), G = kUVWarps / wps
  // columns at a time
  int nseg = 0;
  for (int r = 0; r < nb; ++r) nseg += seg_hi[r] - seg_lo[r];
  const int avg = (nseg + nb - 1) / nb;
  int g_min = 1;
  while (g_min < kUVWarps && g_min < nb) g_min *= 2;
  int wps = 1;
  while (wps < kUVWarps / g_min && kUVBatch * wps < avg) wps *= 2;
  const int G = kUVWarps / wps, wi = warp % wps;
  for (int base = 0; base < nb; base += G) {
    const int r = base + warp / wps;  // this warp's column in the tile
    float acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = 0.f;
    if (r < nb) {
      const int c = b0 + r, s0 = seg_lo[r], n = seg_hi[r] - s0, row = row_of[r];
      const float* lse = p.partial_lse + size_t(s0) * p.heads + row;
      const float* po = p.partial_o + size_t(s0) * p.heads * kLatent + size_t(row) * kLatent + 16 * lane;
      const size_t seg_stride = size_t(p.heads) * kLatent;
      // the first batch of rows is requested together with the lse values
      float4 v[kUVBatch][4];
#pragma unroll
      for (int u = 0; u < kUVBatch; ++u) {
        const int i = wi + u * wps;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          v[u][q] = i < n ? reinterpret_cast<const float4*>(po + i * seg_stride)[q] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      // max and sum of exp(lse - max) over the segments, kLseRegs x 32 lse
      // values per pass (requested together); with at most that many
      // segments, lane l keeps exp(lse_{32 j + l} - max) in e[j] for the weights
      constexpr int kLseRegs = 4;
      float mx = -INFINITY, z = 0.f, e[kLseRegs] = {};
      for (int i0 = 0; i0 < n; i0 += 32 * kLseRegs) {
        float l[kLseRegs];
#pragma unroll
        for (int j = 0; j < kLseRegs; ++j) {
          const int i = i0 + 32 * j + lane;
          l[j] = i < n ? lse[size_t(i) * p.heads] : -INFINITY;
        }
        float m2 = l[0];
#pragma unroll
        for (int j = 1; j < kLseRegs; ++j) m2 = fmaxf(m2, l[j]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m2 = fmaxf(m2, __shfl_xor_sync(0xffffffffu, m2, o));
        m2 = fmaxf(m2, mx);
        if (m2 != -INFINITY) {
          float zs = 0.f;
#pragma unroll
          for (int j = 0; j < kLseRegs; ++j) {
            e[j] = expf(l[j] - m2);
            zs += e[j];
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) zs += __shfl_xor_sync(0xffffffffu, zs, o);
          z = (mx == -INFINITY ? 0.f : z * expf(mx - m2)) + zs;
          mx = m2;
        }
      }
      if (wi == 0 && lane == 0 && p.lse_out)
        p.lse_out[size_t(c) * p.heads_w + h] = mx != -INFINITY ? mx + logf(z) : -INFINITY;
      if (mx != -INFINITY) {
        const float inv_z = 1.f / z;
        // segments wi, wi + wps, ..., kUVBatch at a time
        for (int k = wi;; ) {
          float w[kUVBatch];
#pragma unroll
          for (int u = 0; u < kUVBatch; ++u) {
            const int i = k + u * wps;
            if (n <= 32 * kLseRegs) {
              float ej = e[0];
#pragma unroll
              for (int j = 1; j < kLseRegs; ++j)
                if ((i >> 5) == j) ej = e[j];
              w[u] = __shfl_sync(0xffffffffu, ej, i & 31) * inv_z;
            } else {
              w[u] = i < n ? expf(lse[size_t(i) * p.heads] - mx) * inv_z : 0.f;
            }
            if (i >= n) w[u] = 0.f;
          }
#pragma unroll
          for (int u = 0; u < kUVBatch; ++u)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              acc[4 * q] = fmaf(w[u], v[u][q].x, acc[4 * q]);
              acc[4 * q + 1] = fmaf(w[u], v[u][q].y, acc[4 * q + 1]);
              acc[4 * q + 2] = fmaf(w[u], v[u][q].z, acc[4 * q + 2]);
              acc[4 * q + 3] = fmaf(w[u], v[u][q].w, acc[4 * q + 3]);
            }
          k += kUVBatch * wps;
          if (k >= n) break;
#pragma unroll
          for (int u = 0; u < kUVBatch; ++u) {
            const int i = k + u * wps;
#pragma unroll
            for (int q = 0; q < 4; ++q)
              v[u][q] = i < n ? reinterpret_cast<const float4*>(po + i * seg_stride)[q] : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
      }
    }
    if (wps == 1) {  // lane l holds latent dims [16 l, 16 l + 16)
      if (r < nb) {
        store_planes<NB>(bsm, r, 16 * lane, acc);
        store_planes<NB>(bsm, r, 16 * lane + 8, acc + 8);
      }
    } else {  // add the wps warps' sums in warp order
      float4* mine = reinterpret_cast<float4*>(xs + warp * kLatent) + 4 * lane;
#pragma unroll
      for (int q = 0; q < 4; ++q) mine[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
      __syncthreads();
      if (wi == 0 && r < nb) {
#pragma unroll 1
        for (int k = 1; k < wps; ++k) {
          const float4* other = reinterpret_cast<const float4*>(xs + (warp + k) * kLatent) + 4 * lane;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 x = other[q];
            acc[4 * q] += x.x;
            acc[4 * q + 1] += x.y;
            acc[4 * q + 2] += x.z;
            acc[4 * q + 3] += x.w;
          }
        }
        store_planes<NB>(bsm, r, 16 * lane, acc);
        store_planes<NB>(bsm, r, 16 * lane + 8, acc + 8);
      }
      __syncthreads();
    }
  }
  // rows past the batch: zeros (their output columns are discarded)
  for (int i = tid; i < (NB - nb) * (kLatent / 8); i += kUVThreads) {
    const float z8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    store_planes<NB>(bsm, nb + i / (kLatent / 8), 8 * (i % (kLatent / 8)), z8);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot, sbase = smem_u32(smem);

  // ---- 2. D = W^UV_h [hi | lo]^T
  bool ok = true;
  if (tid == 0) {
    ok = mbar_wait(w_full, 0, abort_flag, kUVWaitNs);
    tc_fence_after();
    if (ok) {
      constexpr uint32_t idesc = idesc_f32acc(128, 2 * NB, false, false, false);
      constexpr uint64_t kDesc = smem_desc(0, 16, 1024, kSwizzle128B);
#pragma unroll
      for (int kk = 0; kk < kLatent / 16; ++kk)
        mma_bf16(tmem, kDesc | desc_addr(sbase + (kk >> 2) * kUVWBlock + (kk & 3) * 32),
                 kDesc | desc_addr(sbase + C::kOffB + (kk >> 2) * C::kBBlock + (kk & 3) * 32), idesc, kk != 0);
      mma_commit(mma_done);
    } else {
      *abort_flag = 1;
    }
  }
  __syncthreads();
  ok = *abort_flag == 0 && mbar_wait(mma_done, 0, abort_flag, kUVWaitNs);
  tc_fence_after();
  if (!ok && tid == 0) set_status(p.status, MLA_ERR_DEVICE_TIMEOUT);

  // ---- 3. thread (warp, lane) of warps 0-3 holds output dim j = 32 warp + lane
  if (ok && warp < 4) {
    const int j = 32 * warp + lane;
    const uint32_t row = uint32_t(32 * warp) << 16;
#pragma unroll
    for (int c = 0; c < NB; c += 8) {
      float vh[8], vl[8];
      tmem_ld8(tmem + row + c, vh);
      tmem_ld8(tmem + row + NB + c, vl);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (c + i < nb) p.out[(size_t(b0 + c + i) * p.heads_w + h) * kVDim + j] = __float2bfloat16_rn(vh[i] + vl[i]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (!ok && tid == 0) {  // let a copy still in flight land before the CTA's shared memory is released
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 20000) {
    }
  }
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int NB>
cudaError_t launch_merge_uv(const CombineUVParams& p, cudaStream_t stream) {
  using C = UVCfg<NB>;
  CUtensorMap mw;
  if (!dc::make_map_2d(&mw, p.W_UV, 2, kLatent, uint64_t(p.heads_w) * kVDim, 64, kVDim, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  static std::atomic<bool> attr[128];  // per device: attributes set (zero-initialised)
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 128 || !attr[dev]) {
    const cudaError_t e =
        cudaFuncSetAttribute(merge_uv_kernel<NB>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(C::kSmem));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 128) attr[dev] = true;
  }
  const int grid = p.heads_w * ((p.batch * p.q_len + NB - 1) / NB);
  return launch_pdl(merge_uv_kernel<NB>, dim3(grid), dim3(kUVThreads), C::kSmem, stream, 1, mw, p);
}

cudaError_t launch_combine_uv(const CombineUVParams& p, cudaStream_t stream) {
  // the largest tile that still gives every SM a CTA; 8 columns when none does
  const int cols = p.batch * p.q_len;
  if (p.heads_w * ((cols + 31) / 32) >= p.sm_count) return launch_merge_uv<32>(p, stream);
  if (p.heads_w * ((cols + 15) / 16) >= p.sm_count) return launch_merge_uv<16>(p, stream);
  return launch_merge_uv<8>(p, stream);
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
