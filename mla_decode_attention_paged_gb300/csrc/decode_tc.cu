// decode_tc.cu -- split-KV MLA decode attention on the sm_100-family tensor
// cores (tcgen05 + TMEM), fed by TMA.
//
// What it computes ("The Weight Absorption Trick"; "Seven Ways LLMs Handle
// Attention", section 5; "Flash-Decoding and FlashInfer"): for one head group
// of one sequence and one contiguous range of its tokens, with
// q_full[h] = [W^UK_h^T q_nope_h | q_pe_h] (576 wide) and the cached rows
// c_t = [latent | RoPE key] (576 wide),
//     s[t][h] = scale * q_full[h] . c_t          (all heads share the row)
//     o_lat[h] = sum_t softmax(s[., h])_t * c_t[0:512]
// and emits o_lat (normalised within the range) with the range's lse.
//
// Orientation: both products are taken transposed so that the 128 tokens of
// a tile are the MMA's M extent and the heads its N extent, so no head is
// padded (16 or 32 heads per CTA):
//     S^T [128 tok x HC]  = C_tile [128 x 576]  * Q^T       (A K-major)
//     O^T [512 x HC]     += C_tile^T [512 x 128] * P^T      (A MN-major)
// Each page is read from HBM once for all heads of the group.
//
// bf16 caches: two shared-memory rings.  The QK ring holds single 64-column
// boxes ([128 tok x 64] SW128, 16 KB); every box is released as soon as its
// four QK MMAs complete, so HBM reads never wait for the softmax.  The PV ring
// holds pairs of latent boxes (128 columns = one O^T chunk) that a second
// producer reads again for the PV product, from L2 (the QK read a few
// microseconds earlier brought the lines there).  A single ring serving both
// products has to keep a whole 147 KB tile resident from its QK until its
// PV, which serialises load -> QK -> softmax -> PV per tile.
// 1-byte caches (INT8 or FP8, 73 KB per tile): one ring of pair slots + RoPE
// slots serves both products; the codes are expanded in place.
//
// Warp roles (288 threads; 256 for 32-head bf16 groups; 352 for 1-byte caches):
//   warp 0     TMA producer: Q of each segment; bf16: QK ring 0 (16 heads:
//              boxes 0, 2, 4, 6, 8 of each tile; 32 heads: all 9 boxes);
//              1-byte caches: the pair and RoPE slots (codes)
//   warp 1     TMEM allocation; lane 0 issues the QK^T MMAs
//   warp 2     PV: lane 0 issues the MMAs (a second issuer keeps the tensor
//              pipe busier than one with these small N = 16/32 MMAs); bf16:
//              the warp also clears the ragged tail rows of the last tile
//   warp 3     bf16, 16 heads: QK ring 1 producer (boxes 1, 3, 5, 7): one
//              thread cannot issue TMA copies fast enough for an SM's share
//              of HBM; bf16, 32 heads: the PV-ring producer
//   warp 8     bf16, 16 heads: the PV-ring producer
//   warps 3, 8-10  INT8 / FP8: expand the TMA-loaded codes in place into
//              fp16 operand tiles
//   warps 4-7  softmax (one thread per token row of S^T) and epilogue
//
// INT8 caches: value = s_t (code - zp_t) per token.  A code v in [-128, 127]
// is expanded to fp16 exactly (bit pattern 0x6400 | (v + 128) is 1152 + v,
// and subtracting 1152 in fp16 is exact), the MMAs run on fp16 operands (Q in
// fp16), and scale and zero point are applied outside the MMAs:
//     s[t][h]   = scale * s_t * (q_h . code_t - zp_t * sum(q_h))
//     o_lat[h]  = (sum_t w_t code_t - sum_t w_t zp_t) / l,  w_t = p_t s_t
// (Leaving the +1152 bias in the operands would make the PV accumulator sum
// ~1152 * sum(w) over thousands of tokens and lose the result to fp32
// cancellation.)
// FP8 caches: value = s_t * e4m3(code), one scale per token.  Every E4M3 value
// is exact in fp16 (see expand_e4m3), so the same fp16 MMAs apply, with no
// zero-point terms:
//     s[t][h]   = scale * s_t * (q_h . e4m3(code_t))
//     o_lat[h]  = sum_t w_t e4m3(code_t) / l,  w_t = p_t s_t
// Every wait is bounded: on timeout the CTA records MLA_ERR_DEVICE_TIMEOUT,
// drains, frees its tensor memory and returns.
#include <atomic>
#include <cuda_fp16.h>

#include "blackwell_ptx.cuh"
#include "decode_common.cuh"
#include "params.cuh"

namespace mla {
namespace {

using namespace ptx;
using namespace dc;

// Nine warps (eleven for 1-byte caches) leave three on one SM sub-partition (16K registers each), which
// caps a thread at 168 registers: enough except for the 32-head bf16 softmax,
// which runs with eight warps and a single QK producer.
constexpr uint32_t kBoxBytes = 16384;           // 128 rows x 128 B (64 bf16)
constexpr uint32_t kPairBytes = 2 * kBoxBytes;  // latent dims [128c, 128c + 128)
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr float kRescaleThreshold = 8.f;        // log2 units
// bf16: the QK read of a page is its first use and the PV read its last; the
// hints keep the lines in L2 between the two and let them go after.
constexpr bool kL2Hints = false;
// bf16: the PV-ring producer reads tile k only once tile k's last QK box has
// landed (when true).  A gated PV read finds its lines in L2 and holds its
// ring slot only for an L2 round trip before the PV MMAs need it.
constexpr bool kPvGate = true;

template <int HC, bool kByte>
struct Cfg {
  static constexpr int kThreads = kByte ? 352 : (HC == 16 ? 288 : 256);
  static constexpr int kQkRings = (!kByte && HC == 16) ? 2 : 1;   // bf16 QK producers (rings)
  static constexpr int kQkSlots = kByte ? 0 : 6;                  // bf16 QK ring slots (single boxes), all rings
  static constexpr int kQkRing = kQkSlots / kQkRings;
  static constexpr int kPvProducerWarp = kQkRings == 2 ? 8 : 3;
  static constexpr int kNumPair = kByte ? 5 : (HC == 16 ? 3 : 2);  // bf16 PV ring / 1-byte shared ring
  static constexpr int kNumRope = kByte ? 2 : 0;
  static constexpr uint32_t kQBytes = 9 * HC * 128;
  static constexpr uint32_t kPBytes = kTile * HC * 2;
  static constexpr uint32_t kOffQk = 0;
  static constexpr uint32_t kOffPair = kOffQk + kQkSlots * kBoxBytes;
  static constexpr uint32_t kOffRope = kOffPair + kNumPair * kPairBytes;
  static constexpr uint32_t kOffQ = kOffRope + kNumRope * kBoxBytes;
  static constexpr uint32_t kOffP = kOffQ + kQBytes;
  static constexpr uint32_t kOffMisc = kOffP + 2 * kPBytes;
  static constexpr uint32_t kMiscBytes = 4096;
  static constexpr uint32_t kSmem = kOffMisc + kMiscBytes + 1024;  // +1024: base alignment slack
  static constexpr uint32_t kTmemCols = HC == 16 ? 128 : 256;      // S^T x2 + O^T x4 = 6 * HC
  static constexpr uint32_t kColS = 0;                             // + buf * HC
  static constexpr uint32_t kColO = 2 * HC;                        // + c * HC
  static_assert(kSmem <= 232448, "dynamic shared memory of one CTA");
  static_assert(kQkRing <= 8 && kNumPair <= 5 && kNumRope <= 2, "barrier arrays");
  static_assert(1024 + 17 * HC * 4 <= kMiscBytes, "barriers, maxima, sums and reciprocal sums");
};

struct Barriers {
  uint64_t full_qk[2][8], empty_qk[2][8];            // bf16 QK rings
  uint64_t full_pair[5], empty_pair[5];              // bf16 PV ring; 1-byte shared ring
  uint64_t full_rope[2], empty_rope[2];              // 1-byte caches
  uint64_t full_i8_pair[5], full_i8_rope[2];         // 1-byte caches: TMA landed, codes not yet expanded
  uint64_t q_full, q_empty, s_full[2], p_full[2], pv_done[2], o_full, o_free, drain[2];
  uint32_t tmem_base;
  int abort;
  int qk_progress;  // bf16: tiles the QK side has finished with (see kPvGate)
};

__device__ __forceinline__ void publish_progress(int* counter, int value) {
  *reinterpret_cast<volatile int*>(counter) = value;
}
// Waits until *counter > k; false on abort or after limit_ns.
__device__ __forceinline__ bool wait_progress(const int* counter, int k, const volatile int* abort,
                                              uint64_t limit_ns) {
  const volatile int* c = counter;
  if (*c > k) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (*c > k) return true;
    if ((i & 63) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > limit_ns) return false;
    }
  }
}

__device__ __forceinline__ void fail(Barriers* B, int* status) {
  B->abort = 1;
  set_status(status, MLA_ERR_DEVICE_TIMEOUT);
}

// kCode: CacheCode (bf16, INT8 or FP8 rows).
// kCausal: multi-token decode (q_len > 1) only, as in the pair kernel.
template <int HC, int kCode, bool kCausal>
__global__ void __launch_bounds__(Cfg<HC, kCode != kCodeBf16>::kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmap_cache, const __grid_constant__ CUtensorMap tmap_q,
                     DecodeParams p) {
  constexpr bool kByte = kCode != kCodeBf16;  // 1-byte codes, expanded to fp16 in shared memory
  constexpr bool kZp = kCode == kCodeInt8;    // per-token zero point (INT8)
  using C = Cfg<HC, kByte>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Barriers* B = reinterpret_cast<Barriers*>(smem + C::kOffMisc);
  // [2][HC][4] maxima, [HC][4] sums of l, [HC][4] sums of corr, [HC] 1 / l
  float* red = reinterpret_cast<float*>(smem + C::kOffMisc + 1024);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr uint32_t kFullCount = 1;  // TMA (bf16) or expansion thread 0 (1-byte caches) completes a slot

  if (threadIdx.x == 0) {
    for (int r = 0; r < C::kQkRings; ++r)
      for (int i = 0; i < C::kQkRing; ++i) {
        mbar_init(&B->full_qk[r][i], 1);
        mbar_init(&B->empty_qk[r][i], 1);
      }
    for (int i = 0; i < C::kNumPair; ++i) {
      mbar_init(&B->full_pair[i], kFullCount);
      mbar_init(&B->empty_pair[i], 1);
      mbar_init(&B->full_i8_pair[i], 1);
    }
    for (int i = 0; i < C::kNumRope; ++i) {
      mbar_init(&B->full_rope[i], kFullCount);
      mbar_init(&B->empty_rope[i], 1);
      mbar_init(&B->full_i8_rope[i], 1);
    }
    mbar_init(&B->q_full, 1);
    mbar_init(&B->q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&B->s_full[i], 1);
      mbar_init(&B->p_full[i], 128);
    }
    mbar_init(&B->pv_done[0], 1);
    mbar_init(&B->pv_done[1], 1);
    mbar_init(&B->o_full, 1);
    mbar_init(&B->o_free, 128);
    mbar_init(&B->drain[0], 1);
    mbar_init(&B->drain[1], 1);
    B->abort = 0;
    B->qk_progress = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmap_cache);
    prefetch_tensormap(&tmap_q);
  }
  if (warp == 1) {
    tmem_alloc(&B->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = B->tmem_base;
  griddep_wait();  // the plan and Q come from the kernel before
  griddep_launch_dependents();

  const int G = p.num_groups, g = blockIdx.x % G, cp = blockIdx.x / G, Cp = gridDim.x / G;
  const long long S = p.status[1];  // effective split count from the plan
  const long long pa = (cp * S) / Cp, pb = ((cp + 1) * S) / Cp;
  const volatile int* abort_flag = &B->abort;
  const int P = p.page_size;

  if ((warp == 0 || (C::kQkRings == 2 && warp == 3)) && lane == 0) {
    // ------------------------------------------------------------ producers
    // bf16, 16 heads: warp 0 fills QK ring 0 with boxes 0, 2, 4, 6, 8 of
    // every tile (and loads Q), warp 3 fills ring 1 with boxes 1, 3, 5, 7:
    // one thread cannot issue TMA copies fast enough to stream an SM's share
    // of HBM and also keep up with the rest of the kernel.
    const int qr = warp == 0 ? 0 : 1;
    TileWalker walk;
    walk.init(p.tile_start, p.seg_base, p.len, p.batch, int(S), pa, pb);
    const uint64_t pol_keep = policy_evict_last();
    auto load = [&](void* dst, int x, int y, uint64_t* bar) {
      if (kL2Hints && !kByte) tma_load_2d_hint(dst, &tmap_cache, x, y, bar, pol_keep);
      else tma_load_2d(dst, &tmap_cache, x, y, bar);
    };
    const uint32_t page_bytes = uint32_t(P) * 128;  // one 64-column box of P rows (bf16)
    uint32_t box_it = 0, pair_it = 0, rope_it = 0, seg = 0;
    TileInfo t, tn;
    TileWalker look = walk;
    TilePages pages, next_pages;
    if (look.next(tn)) next_pages.fetch(p, tn);
    bool ok = true;
    while (ok && walk.next(t)) {
      pages = next_pages;
      if (look.next(tn)) next_pages.fetch(p, tn);
      if (t.first && qr == 0) {
        if (seg > 0 && !(ok = mbar_wait(&B->q_empty, (seg - 1) & 1, abort_flag, kWaitLimitNs))) break;
        mbar_arrive_expect_tx(&B->q_full, C::kQBytes);
        const int qrow = t.b * p.heads + g * HC;
        for (int j = 0; j < 9; ++j) tma_load_2d(smem + C::kOffQ + j * HC * 128, &tmap_q, 64 * j, qrow, &B->q_full);
        ++seg;
      }
      const int npg = pages.npg;
      int rows[kTile / 16];
      pages.rows(p, rows);
      if constexpr (!kByte) {
        // the tile's boxes j = qr, qr + 2, ...: latent columns [64j, 64j + 64), box 8 the RoPE key
        for (int j = qr; j < 9; j += C::kQkRings, ++box_it) {
          const uint32_t slot = box_it % C::kQkRing;
          if (!(ok = mbar_wait(&B->empty_qk[qr][slot], ((box_it / C::kQkRing) & 1) ^ 1, abort_flag, kWaitLimitNs)))
            break;
          uint8_t* dst = smem + C::kOffQk + (qr * C::kQkRing + slot) * kBoxBytes;
          mbar_arrive_expect_tx(&B->full_qk[qr][slot], npg * page_bytes + (p.inject_wait_timeout && box_it == 0 ? 16 : 0));
#pragma unroll 1
          for (int i = 0; i < npg; ++i) load(dst + i * page_bytes, 64 * j, rows[i], &B->full_qk[qr][slot]);
        }
      } else {
        for (int c = 0; c < 4; ++c, ++pair_it) {
          const uint32_t slot = pair_it % C::kNumPair;
          if (!(ok = mbar_wait(&B->empty_pair[slot], ((pair_it / C::kNumPair) & 1) ^ 1, abort_flag, kWaitLimitNs)))
            break;
          // int8 codes of columns [128c, 128c + 128) into the slot's back half, as two [128 x 64 B] blocks
          uint8_t* dst = smem + C::kOffPair + slot * kPairBytes;
          mbar_arrive_expect_tx(&B->full_i8_pair[slot], npg * page_bytes + (p.inject_wait_timeout && pair_it == 0 ? 16 : 0));
#pragma unroll 1
          for (int i = 0; i < npg; ++i) {
            load(dst + kBoxBytes + i * P * 64, 128 * c, rows[i], &B->full_i8_pair[slot]);
            load(dst + kBoxBytes + 8192 + i * P * 64, 128 * c + 64, rows[i], &B->full_i8_pair[slot]);
          }
        }
        if (!ok) break;
        const uint32_t slot = rope_it % C::kNumRope;
        if (!(ok = mbar_wait(&B->empty_rope[slot], ((rope_it / C::kNumRope) & 1) ^ 1, abort_flag, kWaitLimitNs)))
          break;
        uint8_t* dst = smem + C::kOffRope + slot * kBoxBytes;
        mbar_arrive_expect_tx(&B->full_i8_rope[slot], npg * P * 64);
#pragma unroll 1
        for (int i = 0; i < npg; ++i) load(dst + 8192 + i * P * 64, kLatent, rows[i], &B->full_i8_rope[slot]);
        ++rope_it;
      }
    }
    if (!ok) fail(B, p.status);
  } else if (!kByte && warp == C::kPvProducerWarp && lane == 0) {
    // ------------------------------------------------------------ PV-ring producer (bf16)
    // Each tile's latent columns again, pair by pair, for the PV product.
    TileWalker walk;
    walk.init(p.tile_start, p.seg_base, p.len, p.batch, int(S), pa, pb);
    const uint64_t pol_last_use = policy_evict_first();
    const uint32_t page_bytes = uint32_t(P) * 128;
    uint32_t pair_it = 0;
    int k = 0;
    TileInfo t, tn;
    TileWalker look = walk;
    TilePages pages, next_pages;
    if (look.next(tn)) next_pages.fetch(p, tn);
    bool ok = true;
    while (ok && walk.next(t)) {
      pages = next_pages;
      if (look.next(tn)) next_pages.fetch(p, tn);
      const int npg = pages.npg;
      int rows[kTile / 16];
      pages.rows(p, rows);
      if (kPvGate && !(ok = wait_progress(&B->qk_progress, k, abort_flag, kWaitLimitNs))) break;
      ++k;
      for (int c = 0; c < 4; ++c, ++pair_it) {
        const uint32_t slot = pair_it % C::kNumPair;
        if (!(ok = mbar_wait(&B->empty_pair[slot], ((pair_it / C::kNumPair) & 1) ^ 1, abort_flag, kWaitLimitNs)))
          break;
        uint8_t* dst = smem + C::kOffPair + slot * kPairBytes;
        mbar_arrive_expect_tx(&B->full_pair[slot], 2 * npg * page_bytes);
#pragma unroll 1
        for (int i = 0; i < npg; ++i)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (kL2Hints)
              tma_load_2d_hint(dst + h * kBoxBytes + i * page_bytes, &tmap_cache, 128 * c + 64 * h, rows[i],
                               &B->full_pair[slot], pol_last_use);
            else
              tma_load_2d(dst + h * kBoxBytes + i * page_bytes, &tmap_cache, 128 * c + 64 * h, rows[i],
                          &B->full_pair[slot]);
          }
      }
    }
    if (!ok) fail(B, p.status);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ QK issuer
    // S^T[k & 1] = C_tile * Q^T, box by box as the data lands.  Before
    // overwriting S^T[k & 1] it waits for the softmax of tile k - 2 (which
    // read it) to finish.  Descriptors advance by one add per MMA.
    TileWalker walk;
    walk.init(p.tile_start, p.seg_base, p.len, p.batch, int(S), pa, pb);
    constexpr uint32_t id_qk = idesc_f32acc(128, HC, false, false, kByte);
    constexpr uint64_t kDescK = smem_desc(0, 16, 1024, kSwizzle128B);  // K-major SW128
    uint32_t k = 0, seg = 0, box_it[2] = {0, 0};
    TileInfo t;
    bool ok = true;
    while (ok && walk.next(t)) {
      if (k >= 2 && !(ok = mbar_wait(&B->p_full[k & 1], ((k - 2) >> 1) & 1, abort_flag, kWaitLimitNs))) break;
      if (t.first && !(ok = mbar_wait(&B->q_full, seg & 1, abort_flag, kWaitLimitNs))) break;
      const uint32_t d_s = tmem + C::kColS + (k & 1) * HC;
      if constexpr (!kByte) {
        for (int j = 0; j < 9; ++j) {
          const int r = j % C::kQkRings;
          const uint32_t slot = box_it[r] % C::kQkRing, par = (box_it[r] / C::kQkRing) & 1;
          ++box_it[r];
          if (!(ok = mbar_wait(&B->full_qk[r][slot], par, abort_flag, kWaitLimitNs))) break;
          if (kPvGate && j == 8) publish_progress(&B->qk_progress, int(k) + 1);
          tc_fence_after();
          const uint64_t a0 = kDescK | desc_addr(sbase + C::kOffQk + (r * C::kQkRing + slot) * kBoxBytes);
          const uint64_t b0 = kDescK | desc_addr(sbase + C::kOffQ + j * HC * 128);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) mma_bf16(d_s, a0 + 2 * kk, b0 + 2 * kk, id_qk, (j | kk) != 0);
          mma_commit(&B->empty_qk[r][slot]);
        }
        if (!ok) break;
      } else {
        for (int c = 0; c < 4; ++c) {
          const uint32_t it = 4 * k + c, slot = it % C::kNumPair;
          if (!(ok = mbar_wait(&B->full_pair[slot], (it / C::kNumPair) & 1, abort_flag, kWaitLimitNs))) break;
          tc_fence_after();
          const uint64_t a0 = kDescK | desc_addr(sbase + C::kOffPair + slot * kPairBytes);
          const uint64_t b0 = kDescK | desc_addr(sbase + C::kOffQ + 2 * c * HC * 128);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) mma_bf16(d_s, a0 + 2 * kk, b0 + 2 * kk, id_qk, (c | kk) != 0);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16(d_s, a0 + kBoxBytes / 16 + 2 * kk, b0 + HC * 128 / 16 + 2 * kk, id_qk, 1);
        }
        if (!ok) break;
        const uint32_t rslot = k % C::kNumRope;
        if (!(ok = mbar_wait(&B->full_rope[rslot], (k / C::kNumRope) & 1, abort_flag, kWaitLimitNs))) break;
        tc_fence_after();
        const uint64_t a0 = kDescK | desc_addr(sbase + C::kOffRope + rslot * kBoxBytes);
        const uint64_t b0 = kDescK | desc_addr(sbase + C::kOffQ + 8 * HC * 128);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_bf16(d_s, a0 + 2 * kk, b0 + 2 * kk, id_qk, 1);
        mma_commit(&B->empty_rope[rslot]);
      }
      mma_commit(&B->s_full[k & 1]);
      if (t.last) {
        mma_commit(&B->q_empty);
        ++seg;
      }
      ++k;
    }
    if (!ok) fail(B, p.status);
    mma_commit(&B->drain[0]);  // every MMA this thread issued completes before teardown
    mbar_wait(&B->drain[0], 0, abort_flag, kWaitLimitNs);
  } else if (warp == 2) {
    // ------------------------------------------------------------ PV issuer
    // O^T[c] (+)= C_tile^T[128c .. 128c + 128) * P^T once the softmax of the
    // tile is done; each pair slot is released as soon as its MMAs complete.
    // The whole warp walks the tiles; lane 0 waits and issues.
    TileWalker walk;
    walk.init(p.tile_start, p.seg_base, p.len, p.batch, int(S), pa, pb);
    constexpr uint32_t id_pv = idesc_f32acc(128, HC, true, true, kByte);
    constexpr uint64_t kDescMN = smem_desc(0, kBoxBytes, 1024, kSwizzle128B);  // MN-major SW128
    constexpr uint64_t kDescP = smem_desc(0, 128, 2048, kSwizzleNone);        // P^T core matrices
    uint32_t k = 0, seg = 0, pair_it = 0;
    TileInfo t;
    bool ok = true;
    while (ok && walk.next(t)) {
      bool w = true;
      if (lane == 0) {
        w = mbar_wait(&B->p_full[k & 1], (k >> 1) & 1, abort_flag, kWaitLimitNs);
        if (w && t.first && seg > 0) w = mbar_wait(&B->o_free, (seg - 1) & 1, abort_flag, kWaitLimitNs);
      }
      if (!(ok = __shfl_sync(0xffffffffu, w, 0))) break;
      const int nk = (t.valid + 15) >> 4;
      const int tail_rows = 16 * nk - t.valid;  // rows the last k-step reads past the sequence's end
      const uint64_t bd = kDescP | desc_addr(sbase + C::kOffP + (k & 1) * C::kPBytes);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        const uint32_t slot = kByte ? (4 * k + c) % C::kNumPair : pair_it % C::kNumPair;
        if constexpr (!kByte) {
          if (lane == 0) w = mbar_wait(&B->full_pair[slot], (pair_it / C::kNumPair) & 1, abort_flag, kWaitLimitNs);
          if (!(ok = __shfl_sync(0xffffffffu, w, 0))) break;
          ++pair_it;
          if (tail_rows) {
            // they meet zero weights in P^T but must be finite: clear them
            // (rows past the loaded pages hold whatever the slot held before)
            uint8_t* base = smem + C::kOffPair + slot * kPairBytes;
            for (int i = lane; i < tail_rows * 16; i += 32)
              *reinterpret_cast<uint4*>(base + ((i >> 3) & 1) * kBoxBytes + (t.valid + (i >> 4)) * 128 +
                                        (i & 7) * 16) = make_uint4(0, 0, 0, 0);
            fence_proxy_async_smem();
            __syncwarp();
          }
        }
        if (lane == 0) {
          tc_fence_after();
          const uint64_t ad = kDescMN | desc_addr(sbase + C::kOffPair + slot * kPairBytes);
          const uint32_t d_o = tmem + C::kColO + c * HC;
          if (nk == 8) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) mma_bf16(d_o, ad + 128 * kk, bd + 16 * kk, id_pv, !(t.first && kk == 0));
          } else {
            for (int kk = 0; kk < nk; ++kk) mma_bf16(d_o, ad + 128 * kk, bd + 16 * kk, id_pv, !(t.first && kk == 0));
          }
          mma_commit(&B->empty_pair[slot]);
        }
      }
      if (!ok) break;
      if (lane == 0) {
        mma_commit(&B->pv_done[k & 1]);
        if (t.last) mma_commit(&B->o_full);
      }
      if (t.last) ++seg;
      ++k;
    }
    if (lane == 0) {
      if (!ok) fail(B, p.status);
      mma_commit(&B->drain[1]);
      mbar_wait(&B->drain[1], 0, abort_flag, kWaitLimitNs);
    }
  } else if (kByte && (warp == 3 || warp >= 8)) {
    if constexpr (kByte) {
      // ------------------------------------------------------------ code expansion
      // Warps 3, 8, 9 and 10 turn each landed [128 x 64 B] code block into a
      // swizzled fp16 operand box.  Pair slots hold the codes of boxes 2c and
      // 2c+1 in their back half: block 0 (at +16 KB) expands into [0, 16 KB)
      // without overlap; block 1 (at +24 KB) overlaps its destination, so all
      // expansion threads read it before any of them writes.  The RoPE slot's
      // block sits at +8 KB and overlaps too.
      constexpr int kRowStep = kConvThreads / 4, kRowsPer = kTile / kRowStep;
      const int ct = (warp == 3 ? 0 : 32 * (warp - 7)) + lane, ch = ct & 3, r0 = ct >> 2;  // rows r0 + kRowStep j
      TileWalker walk;
      walk.init(p.tile_start, p.seg_base, p.len, p.batch, int(S), pa, pb);
      uint32_t pair_it = 0, rope_it = 0;
      TileInfo t;
      bool ok = true;
      auto read_block = [&](const uint8_t* src, uint4 (&v)[kRowsPer]) {
#pragma unroll
        for (int j = 0; j < kRowsPer; ++j)
          v[j] = *reinterpret_cast<const uint4*>(src + (r0 + kRowStep * j) * 64 + ch * 16);
      };
      // rows at and past the tile's valid length are written as zeros: PV reads
      // them (with zero weight) up to the next multiple of 16, and a code there
      // is whatever the cache page holds past the sequence -- for FP8 possibly
      // a NaN pattern, and 0 * NaN would reach the output
      auto write_block = [&](const uint4 (&v)[kRowsPer], uint8_t* dst, int valid) {
        if (valid >= kTile) {  // a full tile (all but a sequence's last): every row is a cached token
#pragma unroll
          for (int j = 0; j < kRowsPer; ++j) {
            const int r = r0 + kRowStep * j;
            uint4 lo, hi;
            if constexpr (kZp) expand_codes(v[j], lo, hi);
            else expand_e4m3(v[j], lo, hi);
            uint8_t* row = dst + r * 128;
            *reinterpret_cast<uint4*>(row + (((2 * ch) ^ (r & 7)) << 4)) = lo;
            *reinterpret_cast<uint4*>(row + (((2 * ch + 1) ^ (r & 7)) << 4)) = hi;
          }
        } else {
#pragma unroll
          for (int j = 0; j < kRowsPer; ++j) {
            const int r = r0 + kRowStep * j;
            uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
            if (r < valid) {
              if constexpr (kZp) expand_codes(v[j], lo, hi);
              else expand_e4m3(v[j], lo, hi);
            }
            uint8_t* row = dst + r * 128;
            *reinterpret_cast<uint4*>(row + (((2 * ch) ^ (r & 7)) << 4)) = lo;
            *reinterpret_cast<uint4*>(row + (((2 * ch + 1) ^ (r & 7)) << 4)) = hi;
          }
        }
      };
      while (ok && walk.next(t)) {
        for (int c = 0; c < 5 && ok; ++c) {
          const bool rope = c == 4;
          const uint32_t it = rope ? rope_it : pair_it, nslot = rope ? C::kNumRope : C::kNumPair;
          const uint32_t slot = it % nslot;
          uint64_t* full_i8 = rope ? &B->full_i8_rope[slot] : &B->full_i8_pair[slot];
          uint8_t* base = smem + (rope ? C::kOffRope + slot * kBoxBytes : C::kOffPair + slot * kPairBytes);
          const bool landed = mbar_wait(full_i8, (it / nslot) & 1, abort_flag, kWaitLimitNs);
          uint4 v[kRowsPer];
          if (!rope) {
            read_block(base + kBoxBytes, v);
            write_block(v, base, t.valid);
          }
          read_block(base + (rope ? 8192 : kBoxBytes + 8192), v);
          // all codes of the overlapping block read before any write; a timeout
          // anywhere stops the expansion threads together
          if (converters_any(!landed)) {
            ok = false;
            break;
          }
          write_block(v, base + (rope ? 0 : kBoxBytes), t.valid);
          fence_proxy_async_smem();
          converters_sync();
          if (ct == 0) mbar_arrive(rope ? &B->full_rope[slot] : &B->full_pair[slot]);
          if (rope) ++rope_it; else ++pair_it;
        }
      }
      if (!ok) fail(B, p.status);
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ softmax / epilogue
    const int q4 = warp - 4, st = threadIdx.x - 128;  // st = token row of S^T = TMEM lane
    const uint32_t lane_off = uint32_t(q4 * 32) << 16;
    TileWalker walk;
    walk.init(p.tile_start, p.seg_base, p.len, p.batch, int(S), pa, pb);
    float m_run[HC], l_run[HC], corr[HC], qsum[HC];
    uint32_t tile_i = 0, seg = 0;
    TileInfo t;
    while (walk.next(t)) {
      const uint32_t buf = tile_i & 1;
      const bool valid = st < t.valid;
      float tok_s = 0.f, tok_z = 0.f;  // 1-byte codes: this row's scale (and INT8 zero point)
      if (kByte) {
        if (kZp && t.first)
#pragma unroll
          for (int h = 0; h < HC; ++h) {
            const float* qs = p.q_sum + (size_t(t.b) * p.heads + g * HC + h) * kQSumParts;
            float s = qs[0];
#pragma unroll
            for (int c = 1; c < kQSumParts; ++c) s += qs[c];
            qsum[h] = s;
          }
        if (valid) {
          const int tok = t.tile * kTile + st;
          const size_t row = size_t(page_of(p, t.b, tok)) * P + tok % P;
          if (kZp) {
            const float2 sz = *reinterpret_cast<const float2*>(p.scale_zero + row * 2);
            tok_s = sz.x;
            tok_z = sz.y;
          } else {
            tok_s = p.scale_zero[row];
          }
        }
      }
      // S^T of this tile; and PV of tile k - 2, which read the P^T buffer
      // this tile writes, must be complete
      bool ok = mbar_wait(&B->s_full[buf], (tile_i >> 1) & 1, abort_flag, kWaitLimitNs);
      if (tile_i >= 2) ok = ok && mbar_wait(&B->pv_done[buf], ((tile_i - 2) >> 1) & 1, abort_flag, kWaitLimitNs);
      tc_fence_after();
      float x[HC];
      if (ok) {
#pragma unroll
        for (int h0 = 0; h0 < HC; h0 += 16) {
          float v[16];
          tmem_ld16(tmem + lane_off + C::kColS + buf * HC + h0, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) x[h0 + i] = v[i];
        }
      }
      const float row_scale = kByte ? p.scale_log2 * tok_s : p.scale_log2;
#pragma unroll
      for (int h = 0; h < HC; ++h) {
        const float raw = kZp ? fmaf(-tok_z, qsum[h], x[h]) : x[h];
        x[h] = valid ? raw * row_scale : -INFINITY;
      }
      if (kCausal && causal_tile(p, t, walk.len_b)) causal_mask<HC>(x, p, g, walk.len_b, t.tile * kTile + st);
      // Running max.  It only has to bound the scores to within
      // kRescaleThreshold (log2 units), so in the common case every thread
      // checks its own scores against it and the 128 threads OR that flag in
      // the barrier they need anyway.  The first tile of a segment, and a
      // tile that breaks the bound, take the exact path: per-head tile max
      // (transpose-reduce in the warp, then across the 4 warps through shared
      // memory) and, where the max moved, a rescale of O^T and l.
      bool over = false;
      if (!t.first) {
#pragma unroll
        for (int h = 0; h < HC; ++h) over |= x[h] > m_run[h] + kRescaleThreshold;
      }
      float alpha[HC];
      bool rescale = false;
      if (t.first || bar_any(over || !ok)) {
        float* rm = red + buf * 4 * HC;
        {
          float tmp[HC];
#pragma unroll
          for (int h = 0; h < HC; ++h) tmp[h] = x[h];
          const float wm = warp_transpose_reduce<HC, true>(tmp, lane);
          if (HC == 32 || !(lane & 1)) rm[(HC == 32 ? lane : lane >> 1) * 4 + q4] = wm;
        }
        if (bar_any(!ok)) break;
#pragma unroll
        for (int h = 0; h < HC; ++h) {
          const float4 m4 = reinterpret_cast<const float4*>(rm)[h];
          const float mt = fmaxf(fmaxf(m4.x, m4.y), fmaxf(m4.z, m4.w));
          if (t.first) {
            m_run[h] = fmaxf(mt, kEmptyRowMax);  // a row masked in the whole tile stays empty
            l_run[h] = 0.f;
            corr[h] = 0.f;
            alpha[h] = 1.f;
          } else if (mt > m_run[h] + kRescaleThreshold) {
            alpha[h] = exp2f(m_run[h] - mt);
            m_run[h] = mt;
            l_run[h] *= alpha[h];
            corr[h] *= alpha[h];
            rescale = true;
          } else {
            alpha[h] = 1.f;
          }
        }
      }
      if (rescale) {
        // uniform across the 128 threads.  QK of this tile may have been
        // issued before PV of the previous one: wait for that PV first.
        const bool ok3 = mbar_wait(&B->pv_done[(tile_i - 1) & 1], ((tile_i - 1) >> 1) & 1, abort_flag, kWaitLimitNs);
        tc_fence_after();
        if (bar_any(!ok3)) break;
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int h0 = 0; h0 < HC; h0 += 16) {
            float v[16];
            const uint32_t a = tmem + lane_off + C::kColO + c * HC + h0;
            tmem_ld16(a, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] *= alpha[h0 + i];
            tmem_st16(a, v);
          }
        tmem_st_wait();
      }
      // probabilities -> P^T (16-bit, MN-major, no swizzle: 8x8 core matrices)
      uint8_t* pt = smem + C::kOffP + buf * C::kPBytes;
#pragma unroll
      for (int h0 = 0; h0 < HC; h0 += 8) {
        uint32_t packed[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int ha = h0 + 2 * i, hb = ha + 1;
          const float pa_ = ex2_ftz(x[ha] - m_run[ha]), pb_ = ex2_ftz(x[hb] - m_run[hb]);
          if constexpr (kByte) {
            const __half wa = __float2half_rn(pa_ * tok_s), wb = __float2half_rn(pb_ * tok_s);
            l_run[ha] += pa_;
            l_run[hb] += pb_;
            if (kZp) {
              corr[ha] = fmaf(__half2float(wa), tok_z, corr[ha]);
              corr[hb] = fmaf(__half2float(wb), tok_z, corr[hb]);
            }
            packed[i] = uint32_t(__half_as_ushort(wa)) | (uint32_t(__half_as_ushort(wb)) << 16);
          } else {
            const __nv_bfloat16 wa = __float2bfloat16_rn(pa_), wb = __float2bfloat16_rn(pb_);
            l_run[ha] += __bfloat162float(wa);
            l_run[hb] += __bfloat162float(wb);
            packed[i] = uint32_t(__bfloat16_as_ushort(wa)) | (uint32_t(__bfloat16_as_ushort(wb)) << 16);
          }
        }
        *reinterpret_cast<uint4*>(pt + (h0 / 8) * 2048 + (st / 8) * 128 + (st % 8) * 16) =
            make_uint4(packed[0], packed[1], packed[2], packed[3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&B->p_full[buf]);
      ++tile_i;
      if (t.last) {
        const bool ok2 = mbar_wait(&B->o_full, seg & 1, abort_flag, kWaitLimitNs);
        tc_fence_after();
        float* rl = red + 8 * HC;   // [HC][4] sums of l
        float* rc = red + 12 * HC;  // [HC][4] sums of corr (INT8)
        {
          const int hw = HC == 32 ? lane : lane >> 1;
          const bool writer = HC == 32 || !(lane & 1);
          float tmp[HC];
#pragma unroll
          for (int h = 0; h < HC; ++h) tmp[h] = l_run[h];
          const float ls = warp_transpose_reduce<HC, false>(tmp, lane);
          if (writer) rl[hw * 4 + q4] = ls;
          if (kZp) {
#pragma unroll
            for (int h = 0; h < HC; ++h) tmp[h] = corr[h];
            const float cs = warp_transpose_reduce<HC, false>(tmp, lane);
            if (writer) rc[hw * 4 + q4] = cs;
          }
        }
        if (bar_any(!ok2)) break;
        // thread h divides for head h once (a division per head in every
        // thread sits on the pipeline's critical path at every segment end)
        float* rinv = red + 16 * HC;  // [HC]
        float ih = 0.f;
        if (st < HC) {
          const float4 l4 = reinterpret_cast<const float4*>(rl)[st];
          const float l = (l4.x + l4.y) + (l4.z + l4.w);
          ih = l > 0.f ? 1.f / l : 0.f;  // 0: a row with no visible token (multi-token decode)
          rinv[st] = ih;
        }
        if (kZp) {
#pragma unroll
          for (int h = 0; h < HC; ++h) {
            const float4 c4 = reinterpret_cast<const float4*>(rc)[h];
            corr[h] = (c4.x + c4.y) + (c4.z + c4.w);
          }
        }
        bar_any(false);
        float inv_l[HC];
#pragma unroll
        for (int j = 0; j < HC / 4; ++j) {
          const float4 v = reinterpret_cast<const float4*>(rinv)[j];
          inv_l[4 * j] = v.x;
          inv_l[4 * j + 1] = v.y;
          inv_l[4 * j + 2] = v.z;
          inv_l[4 * j + 3] = v.w;
        }
        float* dst = p.partial_o + (size_t(t.seg) * p.heads + g * HC) * kLatent;
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int h0 = 0; h0 < HC; h0 += 16) {
            float v[16];
            tmem_ld16(tmem + lane_off + C::kColO + c * HC + h0, v);
#pragma unroll
            for (int i = 0; i < 16; ++i)
              dst[(h0 + i) * kLatent + c * 128 + st] = (kZp ? v[i] - corr[h0 + i] : v[i]) * inv_l[h0 + i];
          }
        tc_fence_before();
        mbar_arrive(&B->o_free);
        if (st < HC) {  // thread h writes head h's lse
          float mh = 0.f;
#pragma unroll
          for (int h = 0; h < HC; ++h)
            if (st == h) mh = m_run[h];
          p.partial_lse[size_t(t.seg) * p.heads + g * HC + st] = ih > 0.f ? (mh - log2f(ih)) * kLn2 : -INFINITY;
        }
        ++seg;
      }
    }
  }
  // ---------------------------------------------------------------- teardown
  __syncthreads();
  if (B->abort) {  // let copies already issued land before the CTA's shared memory is released
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 20000) {
    }
  }
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
}

// ----- host side: tensor maps and launch ---------------------------------------
template <int HC, int kCode>
cudaError_t launch_tc(const DecodeParams& p, int grid, cudaStream_t stream) {
  constexpr bool kByte = kCode != kCodeBf16;
  using C = Cfg<HC, kByte>;
  CUtensorMap mc, mq;
  const uint64_t rows = uint64_t(p.num_pages) * p.page_size;
  if (!make_map_2d(&mc, p.cache, kByte ? 1 : 2, kRow, rows, 64, p.page_size,
                   kByte ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  // q_full holds bf16 (or, for 1-byte caches, fp16) values; TMA moves 2-byte elements either way
  if (!make_map_2d(&mq, p.q_full, 2, kRow, uint64_t(p.batch) * p.heads, 64, HC, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  static std::atomic<bool> attr[128];  // per device: attributes set (zero-initialised)
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 128 || !attr[dev]) {
    for (auto* k : {decode_tc_kernel<HC, kCode, false>, decode_tc_kernel<HC, kCode, true>}) {
      const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(C::kSmem));
      if (e != cudaSuccess) return e;
    }
    if (dev >= 0 && dev < 128) attr[dev] = true;
  }
  auto* kernel = p.q_len > 1 ? decode_tc_kernel<HC, kCode, true> : decode_tc_kernel<HC, kCode, false>;
  return launch_pdl(kernel, dim3(grid), dim3(C::kThreads), C::kSmem, stream, 1, mc, mq, p);
}

}  // namespace

// Head-group size the attention kernel uses for `heads` query heads (1-byte
// caches: 16, the expansion warps' register budget).
int decode_head_group(int heads, bool byte_cache) { return (!byte_cache && heads % 32 == 0) ? 32 : 16; }

cudaError_t launch_decode_tc(const DecodeParams& p, int hc, int code, int grid, cudaStream_t stream) {
  if (code == kCodeInt8) return launch_tc<16, kCodeInt8>(p, grid, stream);
  if (code == kCodeE4m3) return launch_tc<16, kCodeE4m3>(p, grid, stream);
  return hc == 16 ? launch_tc<16, kCodeBf16>(p, grid, stream) : launch_tc<32, kCodeBf16>(p, grid, stream);
}

}  // namespace mla
