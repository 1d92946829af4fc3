// decode_common.cuh -- pieces shared by the attention kernels: the softmax
// warps' reductions, page lookups and TMA tensor-map construction.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>

#include "params.cuh"

namespace mla {
namespace dc {

__device__ __forceinline__ bool bar_any(bool pred) {  // OR over the 128 softmax threads (named barrier 1)
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(uint32_t(pred))
      : "memory");
  return r != 0;
}

// Reduces N (16 or 32) values per lane over the 32 lanes of a warp with
// log2(32) exchange rounds in which every lane keeps half of its values and
// trades the other half (N - 1 shuffles instead of 5 N).  Returns, in every
// lane, the reduction of value index h = lane >> (32 / N - 1)... that is
// h = lane / 2 for N = 16 (lanes 2h and 2h + 1) and h = lane for N = 32.
template <int N, bool kMax>
__device__ __forceinline__ float warp_transpose_reduce(float (&v)[N], int lane) {
  static_assert(N == 16 || N == 32, "16 or 32 values per lane");
#pragma unroll
  for (int w = N / 2, o = 16; w >= 1; w >>= 1, o >>= 1) {
    const bool upper = lane & o;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float keep = upper ? v[i + w] : v[i];
      const float send = upper ? v[i] : v[i + w];
      const float got = __shfl_xor_sync(0xffffffffu, send, o);
      v[i] = kMax ? fmaxf(keep, got) : keep + got;
    }
  }
  if (N == 16) {
    const float got = __shfl_xor_sync(0xffffffffu, v[0], 1);
    v[0] = kMax ? fmaxf(v[0], got) : v[0] + got;
  }
  return v[0];
}

// 2^x with the hardware approximation (relative error about 2^-22, far
// below the bf16 rounding the probabilities get next); flushes subnormal
// results to zero, which only affects weights below 2^-126.
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two fp32 values rounded to fp16 (round to nearest even, magnitudes past
// 65504 saturate to it) in one 32-bit word, `lo` in the low half.
__device__ __forceinline__ uint32_t pack_f16x2_sat(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float2 unpack_f16x2(uint32_t v) {
  return __half22float2(*reinterpret_cast<const __half2*>(&v));
}

// Multi-token decode ("The Architecture of Memory", "Speculative Decoding"
// and "Tree Attention Verification": the new tokens see the history and the
// new tokens before them).  Row h of head group g is query token
// (g HC + h) / heads_w, at position len - q_len + that token; the score of
// cache position `pos` is masked for every row whose position is below pos.
// Only tiles that reach past position len - q_len need it.
__device__ __forceinline__ bool causal_tile(const DecodeParams& p, const TileInfo& t, int len) {
  return p.q_len > 1 && t.tile * kTile + t.valid > len - p.q_len + 1;
}
template <int HC>
__device__ __forceinline__ void causal_mask(float (&x)[HC], const DecodeParams& p, int g, int len, int pos) {
  const int first = len - p.q_len;  // position of query token 0
#pragma unroll
  for (int h = 0; h < HC; ++h)
    if (pos > first + (g * HC + h) / p.heads_w) x[h] = -INFINITY;
}
// Running max of a row with no unmasked score yet: finite, so that
// exp2(x - max) of a masked score is 0 rather than NaN, and below any score.
constexpr float kEmptyRowMax = -1e30f;

// Physical page of token `tok` of sequence b (range-checked; out-of-range
// entries are reported and replaced by page 0 to stay in bounds).
__device__ __forceinline__ int page_of(const DecodeParams& p, int b, int tok) {
  int pg = p.block_table[size_t(b) * p.max_pages + tok / p.page_size];
  if (pg < 0 || pg >= p.num_pages) {
    set_status(p.status, MLA_ERR_DEVICE_BOUNDS);
    pg = 0;
  }
  return pg;
}

// Reports an out-of-range page id (kept out of line: rare, and called from
// several warp roles' hot loops).
static __device__ __noinline__ void report_bad_page(int* status) { set_status(status, MLA_ERR_DEVICE_BOUNDS); }

// Physical pages of one tile, loaded a tile before they are needed: a
// producer that read the block table just in time would stall a full global
// load latency at every tile.  Checked (and clamped to page 0) at use.
struct TilePages {
  int raw[kTile / 16];
  int npg;
  __device__ __forceinline__ void fetch(const DecodeParams& p, const TileInfo& a) {
    npg = (a.valid + p.page_size - 1) / p.page_size;
    const int* bt = p.block_table + size_t(a.b) * p.max_pages + a.tile * (kTile / p.page_size);
#pragma unroll
    for (int i = 0; i < kTile / 16; ++i) raw[i] = i < npg ? __ldg(bt + i) : 0;
  }
  // first cache row (page * P) of each page of the tile into rows[0, npg)
  __device__ __forceinline__ void rows(const DecodeParams& p, int (&r)[kTile / 16]) const {
    bool bad = false;
#pragma unroll
    for (int i = 0; i < kTile / 16; ++i) {
      const bool out = uint32_t(raw[i]) >= uint32_t(p.num_pages);
      bad |= out;
      r[i] = (out ? 0 : raw[i]) * p.page_size;
    }
    if (bad) report_bad_page(p.status);
  }
};

// ----- 1-byte caches: codes expanded to fp16 operands ------------------------
// 1-byte caches: four warps (128 threads) expand the codes, named barrier 2
constexpr int kConvThreads = 128;
__device__ __forceinline__ bool converters_any(bool pred) {  // OR over the expansion threads (barrier 2)
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 2, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(uint32_t(pred)), "n"(kConvThreads)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void converters_sync() { asm volatile("bar.sync 2, %0;" ::"n"(kConvThreads) : "memory"); }

// 16 int8 codes -> 16 fp16 values equal to the codes, as two 16-byte halves.
__device__ __forceinline__ uint32_t codes_to_half2(uint32_t biased_bits) {  // (1152 + a, 1152 + b) -> (a, b)
  const __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&biased_bits), __floats2half2_rn(1152.f, 1152.f));
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ void expand_codes(uint4 v, uint4& lo, uint4& hi) {
  const uint32_t w[4] = {v.x ^ 0x80808080u, v.y ^ 0x80808080u, v.z ^ 0x80808080u, v.w ^ 0x80808080u};
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    o[2 * i] = codes_to_half2(__byte_perm(w[i], 0x64646464u, 0x4140));      // bytes 0,1 -> 0x64xx 0x64xx
    o[2 * i + 1] = codes_to_half2(__byte_perm(w[i], 0x64646464u, 0x4342));  // bytes 2,3
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// 16 E4M3 codes -> 16 fp16 values equal to the codes' values (every E4M3
// value is exact in fp16: at most 4 significant bits, magnitudes 2^-9..448),
// one conversion instruction per pair; byte k of each word becomes half k.
__device__ __forceinline__ uint32_t e4m3x2_to_half2(uint32_t two_codes) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(uint16_t(two_codes)));
  return r;
}
__device__ __forceinline__ void expand_e4m3(uint4 v, uint4& lo, uint4& hi) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    o[2 * i] = e4m3x2_to_half2(w[i]);            // bytes 0,1
    o[2 * i + 1] = e4m3x2_to_half2(w[i] >> 16);  // bytes 2,3
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// Dequantisation of 16 expanded codes (8 fp16 pairs equal to the codes'
// values) in place: each becomes code * scale + nzs (nzs = -zero point x
// scale; 0 for FP8), evaluated with one fp32 fused multiply-add and rounded
// once to fp16 (magnitudes past 65504 saturate to it).
__device__ __forceinline__ uint32_t dequant_half2(uint32_t codes, float scale, float nzs) {
  const float2 f = unpack_f16x2(codes);
  return pack_f16x2_sat(fmaf(f.x, scale, nzs), fmaf(f.y, scale, nzs));
}
__device__ __forceinline__ void dequant16(uint4& lo, uint4& hi, float scale, float nzs) {
  lo = make_uint4(dequant_half2(lo.x, scale, nzs), dequant_half2(lo.y, scale, nzs), dequant_half2(lo.z, scale, nzs),
                  dequant_half2(lo.w, scale, nzs));
  hi = make_uint4(dequant_half2(hi.x, scale, nzs), dequant_half2(hi.y, scale, nzs), dequant_half2(hi.z, scale, nzs),
                  dequant_half2(hi.w, scale, nzs));
}

// ----- host side: tensor maps ----------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
  // resolved once; the initialisation of a function-local static is thread-safe
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// 2-D map over a row-major [rows, inner] tensor of 1- or 2-byte elements.
inline bool make_map_2d(CUtensorMap* m, const void* base, int elem_bytes, uint64_t inner, uint64_t rows,
                        uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * elem_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace dc
}  // namespace mla
