// append.cu -- write new tokens into the paged latent cache.
//
// "The Architecture of Memory", decode phase: the new token's key/value state
// is appended to the cache; in MLA that state is one 576-wide row, the latent
// c_t plus the decoupled RoPE key ("Beyond the Attention Bottleneck", "The RoPE
// Compatibility Problem": only the positional key carries RoPE, rotated here
// once at its position).  Pages are found through the page table
// ("PagedAttention: Virtual Memory for LLMs").  1-byte caches quantise the
// row per token ("KV Cache Optimization", section 3; "The Architecture of
// Memory", KIVI section): INT8 with an asymmetric min/max scale and zero
// point, FP8 (E4M3) with one scale that maps the row's largest magnitude to
// 448, the format's largest finite value.
#include "blackwell_ptx.cuh"
#include "params.cuh"

namespace mla {


// Two fp32 values to E4M3 codes (round to nearest even, saturating to
// +-448), first value in the low byte.
__device__ __forceinline__ uint32_t e4m3x2_rn_sat(float first, float second) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(second), "f"(first));
  return r;
}

// One warp per token.  Lane l owns latent values [16l, 16l + 16) and RoPE pair l.
template <int kCode>
__global__ void __launch_bounds__(256) append_kernel(AppendParams p) {
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int i = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (i >= p.n_tokens) return;
  const int b = p.chunk > 0 ? i / p.chunk : p.seq_ids[i];
  // 64-bit: a length near the int32 limits must not wrap into a valid position
  const long long pos64 = p.chunk > 0 ? (long long)p.seq_lens[b] - p.chunk + i % p.chunk : p.positions[i];
  bool ok = b >= 0 && b < p.num_seqs && pos64 >= 0 && pos64 / p.page_size < p.max_pages;
  const int pos = int(pos64);  // in [0, max_pages * P) once ok
  int page = -1;
  if (ok) {
    page = p.block_table[size_t(b) * p.max_pages + pos / p.page_size];
    ok = page >= 0 && page < p.num_pages;
  }
  if (!ok) {
    if (lane == 0) set_status(p.status, MLA_ERR_DEVICE_BOUNDS);
    return;
  }
  const size_t row = size_t(page) * p.page_size + pos % p.page_size;

  // latent part: 16 bf16 per lane, two 16-byte loads
  const uint4* src = reinterpret_cast<const uint4*>(p.c_kv + size_t(i) * kLatent) + 2 * lane;
  uint4 c0 = src[0], c1 = src[1];

  // RoPE pair `lane`: angle = pos * theta^(-2 lane / 64) in fp64 (up to
  // ~2^31 rad), reduced modulo 2 pi in fp64 to [-pi, pi]; sine, cosine and
  // the rotation then in fp32 ahead of the one rounding to bf16.  A full
  // fp64 sincos per lane kept the few SMs an append runs on busy for
  // microseconds (the fp64 units are a small fraction of this part's), and
  // the reduced fp32 result stays far inside the bf16 rounding.
  const __nv_bfloat162 kp = reinterpret_cast<const __nv_bfloat162*>(p.k_pe + size_t(i) * kRope)[lane];
  __nv_bfloat162 kr = kp;
  if (p.rope_theta > 0.0) {
    constexpr double kTwoPi = 6.283185307179586476925286766559, kInvTwoPi = 0.15915494309189533576888376337251;
    const double ang = __dmul_rn(double(pos), p.inv_freq[lane]);
    const double turns = rint(__dmul_rn(ang, kInvTwoPi));
    const float red = float(__fma_rn(-turns, kTwoPi, ang));
    float sn, cs;
    sincosf(red, &sn, &cs);
    const float x0 = __low2float(kp), x1 = __high2float(kp);
    kr = __floats2bfloat162_rn(fmaf(x0, cs, -x1 * sn), fmaf(x0, sn, x1 * cs));
  }

  if constexpr (kCode == kCodeBf16) {
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.cache) + row * kRow;
    reinterpret_cast<uint4*>(dst)[2 * lane] = c0;
    reinterpret_cast<uint4*>(dst)[2 * lane + 1] = c1;
    reinterpret_cast<__nv_bfloat162*>(dst + kLatent)[lane] = kr;
  } else {
    // the row's 576 bf16 values, as exact fp32
    float v[18];
    const __nv_bfloat162* c0h = reinterpret_cast<const __nv_bfloat162*>(&c0);
    const __nv_bfloat162* c1h = reinterpret_cast<const __nv_bfloat162*>(&c1);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[2 * j] = __low2float(c0h[j]);
      v[2 * j + 1] = __high2float(c0h[j]);
      v[8 + 2 * j] = __low2float(c1h[j]);
      v[8 + 2 * j + 1] = __high2float(c1h[j]);
    }
    v[16] = __low2float(kr);
    v[17] = __high2float(kr);
    if constexpr (kCode == kCodeE4m3) {
      float a = 0.f;
#pragma unroll
      for (int j = 0; j < 18; ++j) a = fmaxf(a, fabsf(v[j]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
      // IEEE fp32, round to nearest even, in the documented order
      float s = __fdiv_rn(a, 448.f);
      if (s == 0.f) s = 1.f;
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        w[j] = e4m3x2_rn_sat(__fdiv_rn(v[4 * j], s), __fdiv_rn(v[4 * j + 1], s)) |
               (e4m3x2_rn_sat(__fdiv_rn(v[4 * j + 2], s), __fdiv_rn(v[4 * j + 3], s)) << 16);
      uint8_t* dst = static_cast<uint8_t*>(p.cache) + row * kRow;
      reinterpret_cast<uint4*>(dst)[lane] = make_uint4(w[0], w[1], w[2], w[3]);
      reinterpret_cast<uint16_t*>(dst + kLatent)[lane] =
          uint16_t(e4m3x2_rn_sat(__fdiv_rn(v[16], s), __fdiv_rn(v[17], s)));
      if (lane == 0) p.scale_zero[row] = s;
      return;
    }
    float lo = 0.f, hi = 0.f;  // the range always includes 0
#pragma unroll
    for (int j = 0; j < 18; ++j) {
      lo = fminf(lo, v[j]);
      hi = fmaxf(hi, v[j]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    // IEEE fp32, round to nearest even, no contraction, in the documented order
    float s = __fdiv_rn(__fsub_rn(hi, lo), 255.f);
    if (s == 0.f) s = 1.f;
    float zp = rintf(__fsub_rn(-128.f, __fdiv_rn(lo, s)));
    zp = fminf(fmaxf(zp, -128.f), 127.f);
    int8_t q[18];
#pragma unroll
    for (int j = 0; j < 18; ++j) {
      float c = __fadd_rn(rintf(__fdiv_rn(v[j], s)), zp);
      c = fminf(fmaxf(c, -128.f), 127.f);
      q[j] = int8_t(int(c));
    }
    int8_t* dst = static_cast<int8_t*>(p.cache) + row * kRow;
    uint4 packed;
    int8_t* pk = reinterpret_cast<int8_t*>(&packed);
#pragma unroll
    for (int j = 0; j < 16; ++j) pk[j] = q[j];
    reinterpret_cast<uint4*>(dst)[lane] = packed;
    char2 tail;
    tail.x = q[16];
    tail.y = q[17];
    reinterpret_cast<char2*>(dst + kLatent)[lane] = tail;
    if (lane == 0) {
      p.scale_zero[row * 2] = s;
      p.scale_zero[row * 2 + 1] = zp;
    }
  }
}

cudaError_t launch_append(const AppendParams& p, int code, cudaStream_t stream) {
  if (p.n_tokens == 0) return cudaSuccess;
  // a decode step appends one token per sequence: one warp per block spreads
  // the fp64 RoPE over as many SMs as there are tokens
  const int warps = p.n_tokens < 2048 ? 1 : 8;
  const int grid = (p.n_tokens + warps - 1) / warps;
  if (code == kCodeInt8) return launch_pdl(append_kernel<kCodeInt8>, dim3(grid), dim3(warps * 32), 0, stream, 1, p);
  if (code == kCodeE4m3) return launch_pdl(append_kernel<kCodeE4m3>, dim3(grid), dim3(warps * 32), 0, stream, 1, p);
  return launch_pdl(append_kernel<kCodeBf16>, dim3(grid), dim3(warps * 32), 0, stream, 1, p);
}

}  // namespace mla
