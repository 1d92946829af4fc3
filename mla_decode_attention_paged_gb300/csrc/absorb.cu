// absorb.cu -- query absorption and the decode work plan.
//
// Query absorption ("The Architecture of Memory", "The Weight Absorption
// Trick"; "Seven Ways LLMs Handle Attention", section 5): because
// q . (W^UK c) = (W^UK^T q) . c, each head's content query is mapped into
// latent space once per step, q_lat = W^UK_h^T q_nope (512 wide), and the
// attention kernel then scores the 576-wide cached rows directly with
// q_full = [q_lat | q_pe].
#include <atomic>
#include <cuda_fp16.h>

#include "blackwell_ptx.cuh"
#include "decode_common.cuh"
#include "params.cuh"

namespace mla {

using namespace ptx;

// The work plan (checked lengths, each sequence's first tile and first
// segment, the effective split count), built by one extra CTA of the
// absorption grid (its first) while the others absorb.
__device__ void compute_plan(const AbsorbParams& p) {
  __shared__ int scan_tmp[32];
  __shared__ int carry;
  if (threadIdx.x == 0) {
    carry = 0;
    if (p.reset_status) *p.status = MLA_OK;
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

// ---------------------------------------------------------------------------
// Absorption on the tensor cores.  Per weight head h the product is a GEMM
// over every query column -- a (sequence, token) pair: multi-token decode and
// prefill have q_len tokens per sequence, whose rows t * heads_w + h share
// head h's weights --
// q_lat^T [512 x cols] = W^UK_h^T [512 x 128] * q_nope_h^T [128 x cols]; a CTA
// takes one 128-row tile of latent dims (the MMA's M) and NB columns (its N):
//   A = W^UK_h[:, m0:m0+128]^T   MN-major (W^UK rows are 512 latent dims long)
//   B = q_nope[c0:c0+NB, h, :]^T K-major  (q_nope rows are 128 content dims)
// both staged by the CTA's threads into 128-byte-swizzled shared memory, eight
// K = 16 MMAs into an fp32 TMEM accumulator, then one thread per latent dim
// rounds its columns to bf16 (fp16 for 1-byte caches) and stores them.
// Part c of q_sum[column][h] is the sum of the rounded values of latent dims
// [64c, 64c + 64) (part 0 also the RoPE part): INT8 caches need the sum of
// exactly the query the tensor cores see (bf16 and FP8 caches do not use
// it).  1-byte caches take q_full in fp16 (their tensor-core path runs on
// fp16 operands); bf16 caches in bf16.
constexpr int kAbsThreads = 128;
constexpr int kAbsMTile = 128;                               // latent dims per CTA
constexpr uint32_t kAbsBlockBytes = kNope * 64 * 2;          // [128 k x 64 m] bf16, one swizzle column block
constexpr uint32_t kAbsWBytes = 2 * kAbsBlockBytes;          // 32 KB
constexpr uint64_t kAbsWaitNs = 2000000000ull;

template <int NB>
struct AbsCfg {
  static constexpr uint32_t kQBox = NB * 128;                // [NB x 64 k] bf16
  static constexpr uint32_t kOffQ = kAbsWBytes;
  static constexpr uint32_t kOffMisc = kOffQ + 2 * kQBox;
  static constexpr uint32_t kSmem = kOffMisc + 64 + NB * 4 * 4 + NB * 4 + 1024;
  static constexpr uint32_t kTmemCols = NB < 32 ? 32 : NB;
};

template <bool kF16, int NB>
__global__ void __launch_bounds__(kAbsThreads) absorb_kernel(AbsorbParams p) {
  using C = AbsCfg<NB>;
  if (blockIdx.x == 0) {  // the first CTA (scheduled first) builds the work plan
    griddep_wait();
    griddep_launch_dependents();
    compute_plan(p);
    return;
  }
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* mma_done = reinterpret_cast<uint64_t*>(smem + C::kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc + 8);
  int* abort_flag = reinterpret_cast<int*>(smem + C::kOffMisc + 12);
  float* red = reinterpret_cast<float*>(smem + C::kOffMisc + 64);  // [NB][4] per-warp sums
  float* rope_sum = red + NB * 4;                                  // [NB]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // column c0 + r is row (c0 + r) * heads_w + h of q_nope, q_full and q_sum
  const int per_head = 4 * ((p.cols + NB - 1) / NB);
  const int tile = blockIdx.x - 1, h = tile / per_head, rem = tile % per_head, mt = rem & 3, b0 = (rem >> 2) * NB;
  const int m0 = mt * kAbsMTile, nb = min(NB, p.cols - b0);
  if (tid == 0) {
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  griddep_wait();
  griddep_launch_dependents();
  // W^UK_h[k][m0 + m]: row k of 128 dims = 16 chunks of 8; chunk j goes to
  // column block j / 8, 16-byte slot (j % 8) ^ (k % 8).  q_nope[b0 + r][h][:]:
  // chunk j of row r goes to K block j / 8, slot (j % 8) ^ (r % 8).  Every
  // load is issued before the first store, so the staging costs one memory
  // round trip.
  constexpr int kWPer = kNope * 16 / kAbsThreads, kQPer = NB * 16 / kAbsThreads;
  uint4 wv[kWPer], qv[kQPer];
#pragma unroll
  for (int u = 0; u < kWPer; ++u) {
    const int i = tid + u * kAbsThreads, k = i >> 4, j = i & 15;
    wv[u] = *reinterpret_cast<const uint4*>(p.W_UK + (size_t(h) * kNope + k) * kLatent + m0 + 8 * j);
  }
#pragma unroll
  for (int u = 0; u < kQPer; ++u) {
    const int i = tid + u * kAbsThreads, r = i >> 4, j = i & 15;
    qv[u] = make_uint4(0, 0, 0, 0);
    if (r < nb) qv[u] = *reinterpret_cast<const uint4*>(p.q_nope + (size_t(b0 + r) * p.heads_w + h) * kNope + 8 * j);
  }
#pragma unroll
  for (int u = 0; u < kWPer; ++u) {
    const int i = tid + u * kAbsThreads, k = i >> 4, j = i & 15;
    *reinterpret_cast<uint4*>(smem + (j >> 3) * kAbsBlockBytes + k * 128 + (((j & 7) ^ (k & 7)) << 4)) = wv[u];
  }
#pragma unroll
  for (int u = 0; u < kQPer; ++u) {
    const int i = tid + u * kAbsThreads, r = i >> 4, j = i & 15;
    *reinterpret_cast<uint4*>(smem + C::kOffQ + (j >> 3) * C::kQBox + r * 128 + (((j & 7) ^ (r & 7)) << 4)) = qv[u];
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot, sbase = smem_u32(smem);
  if (tid == 0) {
    constexpr uint32_t idesc = idesc_f32acc(128, NB, true, false, false);
    constexpr uint64_t kDescA = smem_desc(0, kAbsBlockBytes, 1024, kSwizzle128B);  // MN-major
    constexpr uint64_t kDescB = smem_desc(0, 16, 1024, kSwizzle128B);              // K-major
#pragma unroll
    for (int kk = 0; kk < kNope / 16; ++kk)
      mma_bf16(tmem, kDescA | desc_addr(sbase + kk * 2048),
               kDescB | desc_addr(sbase + C::kOffQ + (kk >> 2) * C::kQBox + (kk & 3) * 32), idesc, kk > 0);
    mma_commit(mma_done);
  }
  __syncwarp();  // lanes 1-31 must not start waiting while lane 0 still issues
  // RoPE part (m-tile 0): eight threads per sequence, eight values (16 bytes) each
  uint16_t* qf = reinterpret_cast<uint16_t*>(p.q_full);
  if (mt == 0) {
    constexpr int kPasses = NB * 8 / kAbsThreads > 0 ? NB * 8 / kAbsThreads : 1;
    uint4 pe[kPasses];
#pragma unroll
    for (int u = 0; u < kPasses; ++u) {
      const int r = (tid >> 3) + u * (kAbsThreads / 8);
      pe[u] = make_uint4(0, 0, 0, 0);
      if (r < nb)
        pe[u] = *reinterpret_cast<const uint4*>(p.q_pe + (size_t(b0 + r) * p.heads_w + h) * kRope + (tid & 7) * 8);
    }
#pragma unroll
    for (int u = 0; u < kPasses; ++u) {
      const int r = (tid >> 3) + u * (kAbsThreads / 8);
      const __nv_bfloat16* x = reinterpret_cast<const __nv_bfloat16*>(&pe[u]);
      uint16_t o[8];
      float rs = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) rs += round_out<kF16>(bf2f(x[e]), &o[e]);
      if (r < nb)
        *reinterpret_cast<uint4*>(qf + (size_t(b0 + r) * p.heads_w + h) * kRow + kLatent + (tid & 7) * 8) =
            *reinterpret_cast<const uint4*>(o);
      if (kF16) {
#pragma unroll
        for (int off = 4; off > 0; off >>= 1) rs += __shfl_xor_sync(0xffffffffu, rs, off);
        if ((tid & 7) == 0 && r < NB) rope_sum[r] = rs;
      }
    }
  }
  const bool ok = mbar_wait(mma_done, 0, abort_flag, kAbsWaitNs);
  tc_fence_after();
  if (ok) {
    // thread (warp, lane) holds latent dim m0 + 32 warp + lane for every sequence
    const int m = m0 + 32 * warp + lane;
#pragma unroll 1
    for (int c = 0; c < NB; c += 16) {
      float v[16];
      tmem_ld16(tmem + (uint32_t(32 * warp) << 16) + c, v);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int r = c + i;
        v[i] = r < nb ? round_out<kF16>(v[i], qf + (size_t(b0 + r) * p.heads_w + h) * kRow + m) : 0.f;
      }
      if (kF16) {  // 1-byte caches: this warp's 32 dims summed per column; lanes 2i, 2i + 1 get column c + i
        const float sum = dc::warp_transpose_reduce<16, false>(v, lane);
        if (!(lane & 1)) red[(c + (lane >> 1)) * 4 + warp] = sum;
      }
    }
  } else {
    set_status(p.status, MLA_ERR_DEVICE_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  // part 2 mt + q of q_sum[b][h]: latent dims [m0 + 64 q, m0 + 64 q + 64), plus the RoPE part in part 0
  if (kF16 && ok)
    for (int i = tid; i < 2 * nb; i += kAbsThreads) {
      const int r = i >> 1, q = i & 1;
      float v = red[r * 4 + 2 * q] + red[r * 4 + 2 * q + 1];
      if (mt == 0 && q == 0) v += rope_sum[r];
      p.q_sum[(size_t(b0 + r) * p.heads_w + h) * kQSumParts + 2 * mt + q] = v;
    }
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <bool kF16, int NB>
cudaError_t launch_absorb_nb(const AbsorbParams& p, cudaStream_t stream) {
  using C = AbsCfg<NB>;
  static std::atomic<bool> attr[128];  // per device: attributes set (zero-initialised)
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 128 || !attr[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(absorb_kernel<kF16, NB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               int(C::kSmem));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 128) attr[dev] = true;
  }
  const int tiles = p.heads_w * 4 * ((p.cols + NB - 1) / NB);
  return launch_pdl(absorb_kernel<kF16, NB>, dim3(tiles + 1), dim3(kAbsThreads), C::kSmem, stream, 1, p);
}

template <bool kF16>
cudaError_t launch_absorb_t(const AbsorbParams& p, cudaStream_t stream) {
  if (p.cols <= 16) return launch_absorb_nb<kF16, 16>(p, stream);
  if (p.cols <= 32) return launch_absorb_nb<kF16, 32>(p, stream);
  if (p.cols <= 64) return launch_absorb_nb<kF16, 64>(p, stream);
  return launch_absorb_nb<kF16, 128>(p, stream);
}

cudaError_t launch_absorb(const AbsorbParams& p, bool fp16_out, cudaStream_t stream) {
  static_assert(kLatent / 64 == kQSumParts, "one q_sum part per 64 latent dims");
  return fp16_out ? launch_absorb_t<true>(p, stream) : launch_absorb_t<false>(p, stream);
}

}  // namespace mla
