// decode_hm.cu -- split-KV MLA decode attention for groups of 128 query rows
// (128 heads; or q_len x heads rows of multi-token decode and prefill; a
// sequence's last group padded when its rows are not a multiple of 128) on
// CTA pairs, with the query rows as the tensor-core MMA's M extent.  Serves
// bf16, INT8 and FP8 caches.
//
// What it computes ("The Weight Absorption Trick"; "Seven Ways LLMs Handle
// Attention", section 5; "Flash-Decoding and FlashInfer"): for 128 rows h of
// one sequence and one contiguous range of its tokens, with
// q_full[h] = [W^UK_h^T q_nope_h | q_pe_h] (576 wide) and the cached rows
// c_t = [latent | RoPE key] (576 wide),
//     s[h][t] = scale * q_full[h] . c_t
//     o_lat[h] = sum_t softmax(s[h, .])_t * c_t[0:512]
// and emits o_lat (normalised within the range) with the range's lse.  All
// 128 rows share every cached tile, so a tile is read once for all of them
// (DeepSeek-V2's 128 heads share one 576-wide latent row: "Seven Ways LLMs
// Handle Attention", section 5).
//
// Layout.  A 128-row group fills the MMA's M extent, so the rows are M and
// the tokens N (the single-CTA and pair kernels, built for 16 / 32 heads,
// put the tokens on M instead).  The two CTAs of a pair split every cached
// row by columns, as in decode_pair.cu: CTA r holds latent columns
// [256 r, 256 r + 256) and RoPE columns [512 + 32 r, + 32).  Tokens go in
// sub-tiles of 64 (half a work-plan tile):
//   QK: S_r [128 x 64] = Q_r [128 x 288] * C_r [64 x 288]^T, partial over the
//       CTA's columns.  Q_r's latent part sits in tensor memory (A operand
//       from TMEM, loaded once per segment), its RoPE part in shared memory;
//       C_r is the sub-tile's boxes read K-major.
//   exchange: each CTA sends its partial scores, in log2 units rounded to
//       fp16, to the other through distributed shared memory (16 KB per
//       sub-tile); both add the same two fp16 values, so both hold the same
//       scores and run the same softmax.
//   softmax: two threads per row, each with half of the sub-tile's tokens;
//       the pair's maxima meet through shared memory, sums stay per thread
//       until the segment's end.  bf16 caches: P goes to shared memory
//       (K-major, 128-byte swizzle), so a score buffer is free as soon as its
//       scores are read and the next sub-tile's exchange can leave before
//       this sub-tile's P is done.  1-byte caches: P is written into tensor
//       memory over its scores (shared memory holds their code ring instead).
//   PV: O_r [128 x 256] += P [128 x 64] * C_r [64 x 256] (B = the same latent
//       boxes read MN-major): each CTA accumulates its own 256 latent
//       columns, in tensor memory for the whole segment.
// Tensor memory (512 columns): Q latent 128, O_r 256, two score buffers of 64.
//
// 1-byte caches (INT8, FP8): the codes land by TMA in a ring of two code
// slots and four warps turn them into fp16 operand boxes of the dequantised
// values ("KV Cache Optimization", section 3: x = s_t (code - zp_t), INT8;
// x = s_t e4m3(code), FP8), each computed in fp32 and rounded once to fp16.
// Q and P are fp16, and from there the sub-tile runs exactly as for a bf16
// cache: the scale and zero point never reach the softmax.
//
// Warp roles (384 threads; 512 for 1-byte caches):
//   warp 0       TMA producer: Q's RoPE part per segment; latent boxes 0-1 and
//                the RoPE box of every sub-tile (1-byte caches: their codes,
//                into the code ring)
//   warp 1       TMEM allocation; lane 0 issues the QK MMAs
//   warp 2       PV: lane 0 issues the MMAs; bf16: the warp first clears
//                the rows past a sequence's end that the last MMA reads
//   warp 3       TMA producer: latent boxes 2-3 (and 1-byte caches' scales)
//   warps 4-11   Q latent into TMEM per segment, exchange, softmax, epilogue:
//                two threads per row, each with half of the sub-tile's tokens
//   warps 12-15  1-byte caches: code expansion and dequantisation
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

constexpr int kRowsG = 128;                       // query rows per group (MMA M)
constexpr int kSub = 64;                          // tokens per sub-tile (MMA N of QK, K of PV)
constexpr int kMaxSlots = 4;                      // barrier arrays of the sub-tile ring
constexpr uint32_t kLatBox = kSub * 128;          // [64 tokens x 64 latent columns] 16-bit, SW128: 8 KB
constexpr uint32_t kOffRopeBox = 4 * kLatBox;     // [64 tokens x 32 RoPE columns] 16-bit, SW64: 4 KB
// 1-byte caches: a code slot holds a sub-tile's 4 latent code blocks [64 x
// 64 B], its RoPE codes [64 x 32 B] and its per-token (scale, zero point) or
// scale
constexpr int kCodeSlots = 2;
constexpr uint32_t kCodeRope = 4 * 4096, kCodeScl = kCodeRope + 64 * 32, kCodeSlotBytes = 19 * 1024;
constexpr uint32_t kXBytes = kRowsG * kSub * 2;   // one sub-tile's partial scores, fp16
constexpr uint32_t kPBytes = kRowsG * kSub * 2;   // one sub-tile's P [128 x 64] 16-bit, K-major SW128
constexpr uint32_t kQRopeBytes = kRowsG * 32 * 2; // [128 rows x 32 RoPE columns] 16-bit, SW64
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr float kRescaleThreshold = 8.f;          // log2 units
constexpr bool kPrefetchNext = true;              // L2 prefetch of the next sub-tile's boxes
// tensor memory columns: Q's 256 latent values (bf16 / fp16 pairs), O_r, S x2
// (1-byte caches write P over its sub-tile's scores)
constexpr uint32_t kColQ = 0, kColO = 128, kColS = 384, kTmemCols = 512;
constexpr int kSoftWarps = 8;                     // softmax warps: two threads per row

// OR over the softmax threads (named barrier 1), and their barrier
__device__ __forceinline__ bool soft_any(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(uint32_t(pred)), "n"(32 * kSoftWarps)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void soft_sync() { asm volatile("bar.sync 1, %0;" ::"n"(32 * kSoftWarps) : "memory"); }

template <bool kByte>
struct HmCfg {
  static constexpr int kThreads = 128 + 32 * kSoftWarps + (kByte ? 128 : 0);
  static constexpr uint32_t kSlotBytes = 36 * 1024;
  // bf16: three operand slots and P in shared memory (PV's A operand); a
  // fourth slot measured 1-4% slower (the smaller shared-memory footprint
  // leaves more L1).  1-byte caches: four operand slots, P over its scores in
  // TMEM, and a ring of two code slots that the copies land in, so that an
  // operand slot is held only from its expansion to its PV (in shared memory
  // P and the code ring do not both fit)
  static constexpr bool kPSmem = !kByte;
  static constexpr int kSlots = kByte ? 4 : 3;
  static constexpr uint32_t kOffQRope = kSlots * kSlotBytes;
  static constexpr uint32_t kOffP = kOffQRope + kQRopeBytes;  // bf16: [2] P buffers (PV's A operand)
  static constexpr uint32_t kOffCode = kOffP + (kPSmem ? 2 * kPBytes : 0);  // 1-byte: [kCodeSlots] code slots
  static constexpr uint32_t kOffX = kOffCode + (kByte ? kCodeSlots * kCodeSlotBytes : 0);  // [2] peer's partials
  static constexpr uint32_t kOffMisc = kOffX + 2 * kXBytes;
  static constexpr uint32_t kSmem = kOffMisc + 512 + 2048 + 1024;  // + barriers, row maxima and sums, alignment slack
  static_assert(kSmem <= 232448, "dynamic shared memory of one CTA");
  static_assert(kSlots <= kMaxSlots, "barrier arrays");
  static_assert(kOffQRope % 1024 == 0 && kOffP % 1024 == 0 && kSlotBytes % 1024 == 0 && kOffCode % 1024 == 0,
                "swizzle atoms, copy alignment");
};

struct HmBarriers {
  uint64_t full[kMaxSlots];    // sub-tile operands ready (bf16: TMA of both producers; 1-byte: expansion)
  uint64_t empty[kMaxSlots];   // PV of the sub-tile done: the slot may be refilled
  uint64_t landed[kCodeSlots], code_empty[kCodeSlots];  // 1-byte: codes landed (TMA); codes read (expansion)
  uint64_t q_full, q_empty, s_full[2], s_free[2], x_full[2], p_full[2], pv_done[2], o_full, o_free, drain[2];
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void fail(HmBarriers* B, int* status) {
  B->abort = 1;
  set_status(status, MLA_ERR_DEVICE_TIMEOUT);
}

// One 64-token half of a work-plan tile (the plan's unit is 128 tokens).
struct SubTile {
  int b, tok0, valid, seg;
  bool first, last;  // first / last sub-tile of its segment
};

struct SubWalker {
  TileWalkerT<true> w;
  TileInfo t;
  bool pending;  // the tile in t still has its second half to come
  __device__ __forceinline__ void init(const DecodeParams& p, long long S, long long pa, long long pb) {
    w.init(p.tile_start, p.seg_base, p.len, p.batch, int(S), pa, pb);
    pending = false;
  }
  __device__ __forceinline__ bool next(SubTile& s) {
    int half = 1;
    if (pending) {
      pending = false;
    } else {
      if (!w.next(t)) return false;
      half = 0;
      pending = t.valid > kSub;
    }
    s.b = t.b;
    s.tok0 = t.tile * kTile + half * kSub;
    s.valid = half ? t.valid - kSub : (t.valid < kSub ? t.valid : kSub);
    s.seg = t.seg;
    s.first = t.first && half == 0;
    s.last = t.last && !pending;
    return true;
  }
  __device__ __forceinline__ int len() const { return w.len_b; }  // length of the current sub-tile's sequence
};

// Cache rows of a sub-tile's boxes (box_rows = min(P, 64) tokens each),
// block-table entries read one sub-tile ahead; checked at use.
struct SubPages {
  int raw[4], off[4], nb;
  __device__ __forceinline__ void fetch(const DecodeParams& p, const SubTile& s, int box_rows) {
    nb = (s.valid + box_rows - 1) / box_rows;
    const int* bt = p.block_table + size_t(s.b) * p.max_pages;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int tk = s.tok0 + i * box_rows;
      raw[i] = i < nb ? __ldg(bt + tk / p.page_size) : 0;
      off[i] = tk % p.page_size;
    }
  }
  __device__ __forceinline__ void rows(const DecodeParams& p, int (&r)[4], bool report) const {
    bool bad = false;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const bool out = i < nb && uint32_t(raw[i]) >= uint32_t(p.num_pages);
      bad |= out;
      r[i] = (out ? 0 : raw[i]) * p.page_size + off[i];
    }
    if (bad && report) report_bad_page(p.status);
  }
};

// kCode: CacheCode; kCausal: multi-token decode (q_len > 1) masks each row's
// later positions on a sequence's last sub-tiles; kPad: rows per sequence
// not a multiple of 128.
template <int kCode, bool kCausal, bool kPad>
__global__ void __launch_bounds__(HmCfg<kCode != kCodeBf16>::kThreads, 1)
    decode_hm_kernel(const __grid_constant__ CUtensorMap tmap_lat, const __grid_constant__ CUtensorMap tmap_rope,
                     const __grid_constant__ CUtensorMap tmap_qrope, DecodeParams p) {
  constexpr bool kByte = kCode != kCodeBf16;
  constexpr bool kZp = kCode == kCodeInt8;
  using C = HmCfg<kByte>;
  extern __shared__ uint8_t smem_raw[];
  // the same offset in both CTAs: the peer's exchange buffers and barriers are found by mapa
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  HmBarriers* B = reinterpret_cast<HmBarriers*>(smem + C::kOffMisc);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kSlots; ++i) {
      mbar_init(&B->full[i], kByte ? 1 : 2);
      mbar_init(&B->empty[i], 1);
    }
    for (int i = 0; i < kCodeSlots; ++i) {
      mbar_init(&B->landed[i], 2);
      mbar_init(&B->code_empty[i], 1);
    }
    mbar_init(&B->q_full, 1 + 32 * kSoftWarps);  // the RoPE part's TMA, and the rows' latent parts
    mbar_init(&B->q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&B->s_full[i], 1);
      mbar_init(&B->x_full[i], 1);  // armed by one local thread; the peer's bytes complete it
      mbar_init(&B->p_full[i], 32 * kSoftWarps);
      mbar_init(&B->pv_done[i], 1);
      mbar_init(&B->s_free[i], 32 * kSoftWarps);  // every softmax thread has read its scores
      mbar_init(&B->drain[i], 1);
    }
    mbar_init(&B->o_full, 1);
    mbar_init(&B->o_free, 32 * kSoftWarps);
    B->abort = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmap_lat);
    prefetch_tensormap(&tmap_rope);
    prefetch_tensormap(&tmap_qrope);
  }
  if (warp == 1) {
    tmem_alloc(&B->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers exist before either sends to the other
  tc_fence_after();
  const uint32_t tmem = B->tmem_base;
  griddep_wait();  // the plan and Q come from the kernel before
  griddep_launch_dependents();

  const int G = p.num_groups, clus = blockIdx.x / 2, g = clus % G, cp = clus / G, Cp = (gridDim.x / 2) / G;
  const long long S = p.status[1];  // effective split count from the plan
  const long long pa = (cp * S) / Cp, pb = ((cp + 1) * S) / Cp;
  const volatile int* abort_flag = &B->abort;
  const int P = p.page_size, box_rows = P < kSub ? P : kSub;
  const int lat0 = 256 * int(rank), rope0 = kLatent + 32 * int(rank);  // this CTA's columns

  if ((warp == 0 || warp == 3) && lane == 0) {
    // ------------------------------------------------------------ producers
    // Two threads share the copies (one cannot issue them fast enough for an
    // SM's share of HBM): warp 0 the latent boxes 0-1 and the RoPE box, warp 3
    // the latent boxes 2-3 (and, for 1-byte caches, the per-token scales).
    const int role = warp == 0 ? 0 : 1;
    const uint32_t sbytes = kZp ? 8 : 4;  // 1-byte caches: scale bytes per token
    SubWalker walk, look;
    walk.init(p, S, pa, pb);
    look = walk;
    SubTile s, sn;
    SubPages cur, nxt;
    bool have_next = look.next(sn);
    if (have_next) nxt.fetch(p, sn, box_rows);
    uint32_t k = 0, seg = 0;
    bool ok = true;
    while (ok && walk.next(s)) {
      cur = nxt;
      have_next = look.next(sn);
      if (have_next) nxt.fetch(p, sn, box_rows);
      if (s.first && role == 0) {
        if (seg > 0 && !(ok = mbar_wait(&B->q_empty, (seg - 1) & 1, abort_flag, kWaitLimitNs))) break;
        mbar_arrive_expect_tx(&B->q_full, kQRopeBytes);
        tma_load_2d(smem + C::kOffQRope, &tmap_qrope, rope0, s.b * p.heads + g * kRowsG, &B->q_full);
        ++seg;
      }
      int rows[4];
      cur.rows(p, rows, role == 0);
      const int nb = cur.nb;
      if (kPrefetchNext && have_next && G == 1) {
        // the next sub-tile's boxes into L2 now, so that its copies, issued
        // once a slot frees, find them there
        int nrows[4];
        nxt.rows(p, nrows, false);
#pragma unroll 1
        for (int i = 0; i < nxt.nb; ++i) {
          tma_prefetch_2d(&tmap_lat, lat0 + 128 * role, nrows[i]);
          tma_prefetch_2d(&tmap_lat, lat0 + 128 * role + 64, nrows[i]);
          if (role == 0) tma_prefetch_2d(&tmap_rope, rope0, nrows[i]);
        }
      }
      const uint32_t rows_bytes = uint32_t(nb * box_rows);
      if constexpr (!kByte) {
        const uint32_t slot = k % C::kSlots;
        if (!(ok = mbar_wait(&B->empty[slot], ((k / C::kSlots) & 1) ^ 1, abort_flag, kWaitLimitNs))) break;
        uint8_t* base = smem + slot * C::kSlotBytes;
        const uint32_t bytes = rows_bytes * (role == 0 ? 128 + 128 + 64 : 128 + 128);
        mbar_arrive_expect_tx(&B->full[slot], bytes + (p.inject_wait_timeout && k == 0 && role == 0 ? 16 : 0));
#pragma unroll 1
        for (int i = 0; i < nb; ++i) {
          for (int q = 2 * role; q < 2 * role + 2; ++q)
            tma_load_2d(base + q * kLatBox + i * box_rows * 128, &tmap_lat, lat0 + 64 * q, rows[i], &B->full[slot]);
          if (role == 0)
            tma_load_2d(base + kOffRopeBox + i * box_rows * 64, &tmap_rope, rope0, rows[i], &B->full[slot]);
        }
      } else {  // into the code ring; the expansion frees a code slot once it has read it
        const uint32_t cs = k % kCodeSlots;
        if (!(ok = mbar_wait(&B->code_empty[cs], ((k / kCodeSlots) & 1) ^ 1, abort_flag, kWaitLimitNs))) break;
        uint8_t* code = smem + C::kOffCode + cs * kCodeSlotBytes;
        const uint32_t bytes = rows_bytes * (role == 0 ? 64 + 64 + 32 : 64 + 64 + sbytes);
        mbar_arrive_expect_tx(&B->landed[cs], bytes + (p.inject_wait_timeout && k == 0 && role == 0 ? 16 : 0));
#pragma unroll 1
        for (int i = 0; i < nb; ++i) {
          for (int q = 2 * role; q < 2 * role + 2; ++q)
            tma_load_2d(code + q * 4096 + i * box_rows * 64, &tmap_lat, lat0 + 64 * q, rows[i], &B->landed[cs]);
          if (role == 0)
            tma_load_2d(code + kCodeRope + i * box_rows * 32, &tmap_rope, rope0, rows[i], &B->landed[cs]);
          else
            bulk_copy_g2s(code + kCodeScl + i * box_rows * sbytes, p.scale_zero + size_t(rows[i]) * (kZp ? 2 : 1),
                          box_rows * sbytes, &B->landed[cs]);
        }
      }
      ++k;
    }
    if (!ok) fail(B, p.status);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ QK issuer
    // S_r[k & 1] = Q_r * C_r^T: 16 MMAs on the latent columns (A = Q's latent
    // part in TMEM), 2 on the RoPE columns (A = Q's RoPE part in shared
    // memory).  Before overwriting S[k & 1] it waits until sub-tile k - 2 is
    // done with the buffer.
    SubWalker walk;
    walk.init(p, S, pa, pb);
    constexpr uint32_t id_qk = idesc_f32acc(kRowsG, kSub, false, false, kByte);
    constexpr uint64_t kDescK = smem_desc(0, 16, 1024, kSwizzle128B);   // K-major SW128 (8-row groups of 1 KB)
    constexpr uint64_t kDescRope = smem_desc(0, 16, 512, kSwizzle64B);  // K-major SW64 (8-row groups of 512 B)
    uint32_t k = 0, seg = 0;
    SubTile s;
    bool ok = true;
    while (ok && walk.next(s)) {
      const uint32_t sb = k & 1, slot = k % C::kSlots;
      // bf16: every softmax thread has read sub-tile k - 2's scores; 1-byte:
      // PV of sub-tile k - 2 has read its P from the buffer
      if (k >= 2 && !(ok = mbar_wait(C::kPSmem ? &B->s_free[sb] : &B->pv_done[sb], ((k - 2) >> 1) & 1, abort_flag,
                                     kWaitLimitNs)))
        break;
      if (s.first && !(ok = mbar_wait(&B->q_full, seg & 1, abort_flag, kWaitLimitNs))) break;
      if (!(ok = mbar_wait(&B->full[slot], (k / C::kSlots) & 1, abort_flag, kWaitLimitNs))) break;
      tc_fence_after();
      const uint32_t d = tmem + kColS + sb * kSub;
      const uint32_t bs = sbase + slot * C::kSlotBytes;
#pragma unroll
      for (int kk = 0; kk < 16; ++kk)
        mma_f16_tmem_a(d, tmem + kColQ + 8 * kk, kDescK | desc_addr(bs + (kk >> 2) * kLatBox + 32 * (kk & 3)), id_qk,
                       kk > 0);
#pragma unroll
      for (int kk = 0; kk < 2; ++kk)
        mma_bf16(d, kDescRope | desc_addr(sbase + C::kOffQRope + 32 * kk),
                 kDescRope | desc_addr(bs + kOffRopeBox + 32 * kk), id_qk, 1);
      mma_commit(&B->s_full[sb]);
      if (s.last) {
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
    // O_r (+)= P * C_r[:, latent] once the softmax of the sub-tile is done;
    // the slot is released when its MMAs complete.
    SubWalker walk;
    walk.init(p, S, pa, pb);
    constexpr uint32_t id_pv = idesc_f32acc(kRowsG, 256, false, true, kByte);
    constexpr uint64_t kDescMN = smem_desc(0, kLatBox, 1024, kSwizzle128B);  // MN-major SW128, 64-column blocks
    constexpr uint64_t kDescP = smem_desc(0, 16, 1024, kSwizzle128B);        // P: K-major SW128, 128-byte rows
    uint32_t k = 0, seg = 0;
    SubTile s;
    bool ok = true;
    while (ok && walk.next(s)) {
      const uint32_t sb = k & 1, slot = k % C::kSlots;
      bool w = true;
      if (lane == 0) {
        w = mbar_wait(&B->p_full[sb], (k >> 1) & 1, abort_flag, kWaitLimitNs);
        if (w && s.first && seg > 0) w = mbar_wait(&B->o_free, (seg - 1) & 1, abort_flag, kWaitLimitNs);
      }
      if (!(ok = __shfl_sync(0xffffffffu, w, 0))) break;
      const int nk = (s.valid + 15) >> 4;
      if (!kByte && 16 * nk > s.valid) {
        // rows between the sequence's end and the last k-step's bound meet
        // zero probabilities but must be finite (they hold whatever the page's
        // tail or the slot's previous use left): clear them in all 4 boxes
        uint8_t* base = smem + slot * C::kSlotBytes;
        const int tail = 16 * nk - s.valid;
        for (int i = lane; i < tail * 32; i += 32)
          *reinterpret_cast<uint4*>(base + ((i >> 3) & 3) * kLatBox + (s.valid + (i >> 5)) * 128 + (i & 7) * 16) =
              make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (lane == 0) {
        tc_fence_after();
        const uint32_t bs = sbase + slot * C::kSlotBytes;
        if constexpr (C::kPSmem) {
          const uint32_t a = sbase + C::kOffP + sb * kPBytes;  // P of the sub-tile in shared memory
          for (int kk = 0; kk < nk; ++kk)
            mma_bf16(tmem + kColO, kDescP | desc_addr(a + 32 * kk), kDescMN | desc_addr(bs + 2048 * kk), id_pv,
                     !(s.first && kk == 0));
        } else {
          const uint32_t a = tmem + kColS + sb * kSub;  // P: columns [0, 32) of the sub-tile's score buffer
          for (int kk = 0; kk < nk; ++kk)
            mma_f16_tmem_a(tmem + kColO, a + 8 * kk, kDescMN | desc_addr(bs + 2048 * kk), id_pv,
                           !(s.first && kk == 0));
        }
        mma_commit(&B->empty[slot]);
        mma_commit(&B->pv_done[sb]);
        if (s.last) mma_commit(&B->o_full);
      }
      if (s.last) ++seg;
      ++k;
    }
    if (lane == 0) {
      if (!ok) fail(B, p.status);
      mma_commit(&B->drain[1]);
      mbar_wait(&B->drain[1], 0, abort_flag, kWaitLimitNs);
    }
  } else if (kByte && warp >= 4 + kSoftWarps) {
    if constexpr (kByte) {
      // ------------------------------------------------------------ code expansion
      // Each landed sub-tile's codes become fp16 operand boxes of the
      // dequantised values in an operand slot: latent block q -> SW128 box q,
      // RoPE codes -> the SW64 box.  A thread covers tokens ct / 4 and
      // ct / 4 + 32 (latent) and ct / 2 (RoPE): nine 16-code chunks, read,
      // dequantised and written one at a time (the latent loop stays rolled:
      // the expansion's code would otherwise crowd the softmax's out of the
      // instruction cache).  Rows at and past the sequence's end are written
      // as zeros (PV reads them with zero weight, and a code or scale there is
      // whatever the page's tail holds).
      const int ct = threadIdx.x - 128 - 32 * kSoftWarps;
      const int ra = ct >> 2, rr = ct >> 1;
      SubWalker walk;
      walk.init(p, S, pa, pb);
      uint32_t k = 0;
      SubTile s;
      bool ok = true;
      while (ok && walk.next(s)) {
        const uint32_t slot = k % C::kSlots, cs = k % kCodeSlots;
        const uint8_t* code = smem + C::kOffCode + cs * kCodeSlotBytes;
        uint8_t* base = smem + slot * C::kSlotBytes;
        // the codes have landed and PV of sub-tile k - kSlots has freed the operand slot
        bool w = mbar_wait(&B->landed[cs], (k / kCodeSlots) & 1, abort_flag, kWaitLimitNs);
        w = w && mbar_wait(&B->empty[slot], ((k / C::kSlots) & 1) ^ 1, abort_flag, kWaitLimitNs);
        if (converters_any(!w)) {
          ok = false;
          break;
        }
        // the three tokens' scale and -zero point x scale (FP8: no zero point)
        float sc[3], nz[3] = {0.f, 0.f, 0.f};
        {
          const float* scl = reinterpret_cast<const float*>(code + kCodeScl);
          const int rows3[3] = {ra, ra + 32, rr};
#pragma unroll
          for (int j = 0; j < 3; ++j) {
            if constexpr (kZp) {
              const float2 a = reinterpret_cast<const float2*>(scl)[rows3[j]];
              sc[j] = a.x;
              nz[j] = -a.y * a.x;
            } else {
              sc[j] = scl[rows3[j]];
            }
          }
        }
#pragma unroll 1
        for (int i = 0; i < 8; ++i) {  // latent chunk i: token ra + 32 (i & 1), block i / 2
          const int c = ct + 128 * i, q = c >> 8, r = (c >> 2) & 63, ch = c & 3;
          const uint4 v = *reinterpret_cast<const uint4*>(code + q * 4096 + r * 64 + ch * 16);
          uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
          if (r < s.valid) {
            if constexpr (kZp) expand_codes(v, lo, hi);
            else expand_e4m3(v, lo, hi);
            dequant16(lo, hi, (i & 1) ? sc[1] : sc[0], (i & 1) ? nz[1] : nz[0]);
          }
          uint8_t* row = base + q * kLatBox + r * 128;  // 128-byte rows, 128-byte swizzle
          *reinterpret_cast<uint4*>(row + (((2 * ch) ^ (r & 7)) << 4)) = lo;
          *reinterpret_cast<uint4*>(row + (((2 * ch + 1) ^ (r & 7)) << 4)) = hi;
        }
        {  // RoPE chunk: token rr
          const int r = rr, ch = ct & 1;
          const uint4 v = *reinterpret_cast<const uint4*>(code + kCodeRope + r * 32 + ch * 16);
          uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
          if (r < s.valid) {
            if constexpr (kZp) expand_codes(v, lo, hi);
            else expand_e4m3(v, lo, hi);
            dequant16(lo, hi, sc[2], nz[2]);
          }
          uint8_t* row = base + kOffRopeBox + r * 64;  // 64-byte rows, 64-byte swizzle
          *reinterpret_cast<uint4*>(row + (((2 * ch) ^ ((r >> 1) & 3)) << 4)) = lo;
          *reinterpret_cast<uint4*>(row + (((2 * ch + 1) ^ ((r >> 1) & 3)) << 4)) = hi;
        }
        fence_proxy_async_smem();
        converters_sync();
        if (ct == 0) {
          mbar_arrive(&B->code_empty[cs]);  // every thread has read its codes
          mbar_arrive(&B->full[slot]);
        }
        ++k;
      }
      if (!ok) fail(B, p.status);
    }
  } else if (warp >= 4 && warp < 4 + kSoftWarps) {
    // ------------------------------------------------------------ Q, exchange, softmax, epilogue
    // Two threads per row: warp 4 + 4c + q covers rows [32 q, 32 q + 32) (its
    // TMEM lane quarter) and the sub-tile's tokens [32 c, 32 c + 32); the
    // pair of threads of a row combine their maxima (and, at the end, their
    // sums) through shared memory.
    const int sw = warp - 4, q4 = sw & 3, c = sw >> 2, tid = threadIdx.x - 128;
    const int h = 32 * q4 + lane;                     // row of the group = TMEM lane
    const uint32_t lane_off = uint32_t(q4 * 32) << 16;
    const int row = g * kRowsG + h;                   // row within the sequence's rows
    // kPad: a sequence's last group is padded (rows not a multiple of 128):
    // its rows past the end run with a zero latent query and write nothing
    // (a separate instantiation: the check cost the unpadded kernel 2-3%)
    const bool live = !kPad || row < p.heads;
    const uint32_t x_local = sbase + C::kOffX + h * (kSub * 2) + c * kSub;  // this thread's half of its row
    const int xr_rot = h & 3;                         // 16-byte pieces rotated by row to spread banks
    const uint32_t peer = rank ^ 1u;
    // [2 sub-tile parities][2 halves][128] partial row maxima; at a segment's
    // end the other parity's half carries the rows' partial sums
    float* red = reinterpret_cast<float*>(smem + C::kOffMisc + 512);
    SubWalker walk;
    walk.init(p, S, pa, pb);
    float m_run = 0.f, l_run = 0.f;
    uint32_t k = 0, seg = 0;
    // Q's latent part for a segment's sequence into TMEM: this thread's 128
    // of the row's 256 latent values.  Every QK MMA of the previous segment
    // has completed: this thread saw the s_full of its last sub-tile.
    auto load_q = [&](const SubTile& t) {
      const uint4* src =
          reinterpret_cast<const uint4*>(p.q_full + (size_t(t.b) * p.heads + row) * kRow + lat0 + 128 * c);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        uint32_t r[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 v = live ? __ldg(src + 8 * j + i) : make_uint4(0, 0, 0, 0);
          r[4 * i] = v.x; r[4 * i + 1] = v.y; r[4 * i + 2] = v.z; r[4 * i + 3] = v.w;
        }
        tmem_st32(tmem + lane_off + kColQ + 64 * c + 32 * j, r);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&B->q_full);
    };
    // Sub-tile kk's partial scores, this thread's 32 in log2 units rounded to
    // fp16, to the peer (into its buffer kk & 1); kept in hx for the sum.
    // The exchange sends fp16 (distributed shared memory moves only ~12-15
    // GB/s per SM here, so its bytes set the pace) and both CTAs add the same
    // two fp16 values, so both hold the same scores.  Sub-tile k + 1's
    // partials leave as soon as sub-tile k's row maxima are known, so that
    // they cross while sub-tile k's probabilities are computed.  That pays
    // because P lives in shared memory: a score buffer is free once its
    // scores are read here, so QK of sub-tile k + 1 does not wait for PV of
    // sub-tile k - 1 (with P written over the scores in TMEM it did, and the
    // early exchange then held back P instead).
    uint32_t hx[16];
    auto send = [&](uint32_t kk) -> bool {
      const uint32_t xb = kk & 1;
      const bool w = mbar_wait(&B->s_full[xb], (kk >> 1) & 1, abort_flag, kWaitLimitNs);
      if (!w) fail(B, p.status);  // carried to the next barrier; the waits after it return at once
      tc_fence_after();
      uint32_t r[32];
      tmem_ld32(tmem + lane_off + kColS + xb * kSub + 32 * c, r);
      if constexpr (C::kPSmem) {
        tc_fence_before();
        mbar_arrive(&B->s_free[xb]);  // QK of sub-tile kk + 2 may overwrite the buffer
      }
#pragma unroll
      for (int i = 0; i < 16; ++i)
        hx[i] = pack_f16x2_sat(__uint_as_float(r[2 * i]) * p.scale_log2, __uint_as_float(r[2 * i + 1]) * p.scale_log2);
      const uint32_t rbar = mapa_shared(smem_u32(&B->x_full[xb]), peer);
      const uint32_t xr = mapa_shared(x_local + xb * kXBytes, peer);
#pragma unroll
      for (int v = 0; v < 4; ++v)
        st_async_v4_b32(xr + (v ^ xr_rot) * 16, hx[4 * v], hx[4 * v + 1], hx[4 * v + 2], hx[4 * v + 3], rbar);
      if (tid == 0) mbar_arrive_expect_tx(&B->x_full[xb], kXBytes);
      return w;
    };
    SubTile s;
    bool have = walk.next(s), sent_ok = true;
    if (have) {
      if (s.first) load_q(s);
      sent_ok = send(0);
    }
    while (have) {
      const uint32_t sb = k & 1;
      // a failed wait is carried to the maxima's barrier below, where all
      // softmax threads leave together (a named barrier must not be left half-way)
      bool ok = sent_ok && mbar_wait_cluster(&B->x_full[sb], (k >> 1) & 1, abort_flag, kWaitLimitNs);
      if (!ok) fail(B, p.status);
      // S = S_0 + S_1 (addition is commutative: both CTAs get the same bits),
      // in log2 units; tokens past the sub-tile's end (and, for multi-token
      // rows, positions after the row's own) are -inf
      const int t0 = 32 * c;
      const int qpos = kCausal ? walk.len() - p.q_len + row / p.heads_w : 0x7fffffff;
      float x[32];
      float mt = -INFINITY;
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const uint4 y = *reinterpret_cast<const uint4*>(smem + C::kOffX + sb * kXBytes + h * (kSub * 2) + c * kSub +
                                                        (v ^ xr_rot) * 16);
        const uint32_t yy[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 a = unpack_f16x2(hx[4 * v + i]), b = unpack_f16x2(yy[i]);
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int j = 8 * v + 2 * i + e, t = t0 + j;
            bool vis = t < s.valid;
            if (kCausal) vis = vis && s.tok0 + t <= qpos;
            x[j] = vis ? (e ? a.y + b.y : a.x + b.x) : -INFINITY;
            mt = fmaxf(mt, x[j]);
          }
        }
      }
      // the row's max over both halves; the buffer of this parity is written
      // again two sub-tiles on, after the next sub-tile's barrier, which the
      // reads below precede
      red[sb * 256 + c * 128 + h] = mt;
      if (soft_any(!ok)) break;
      mt = fmaxf(mt, red[sb * 256 + (c ^ 1) * 128 + h]);
      // the next sub-tile's partial scores to the peer (and, for a new
      // segment, its Q first: every QK MMA of this segment is complete)
      SubTile sn;
      const bool have_next = walk.next(sn);
      if (C::kPSmem && have_next) {
        if (sn.first) load_q(sn);
        sent_ok = send(k + 1);
      }
      // running max: it only has to bound the row's scores within
      // kRescaleThreshold; the first sub-tile of a segment sets it, a sub-tile
      // that breaks the bound raises it and rescales O and l (both threads of
      // a row take the same decision from the same numbers)
      float alpha = 1.f;
      bool rescale = false;
      if (s.first) {
        m_run = fmaxf(mt, kEmptyRowMax);  // a row masked in the whole sub-tile stays empty
        l_run = 0.f;
      } else if (mt > m_run + kRescaleThreshold) {
        alpha = exp2f(m_run - mt);
        m_run = mt;
        l_run *= alpha;
        rescale = true;
      }
      if (__any_sync(0xffffffffu, rescale)) {
        // PV of the previous sub-tile must be complete before O is rescaled:
        // this thread's 128 of the row's 256 columns
        const bool ok3 = mbar_wait(&B->pv_done[(k - 1) & 1], ((k - 1) >> 1) & 1, abort_flag, kWaitLimitNs);
        tc_fence_after();
        if (__all_sync(0xffffffffu, ok3) && !*abort_flag) {
#pragma unroll 1
          for (int j = 0; j < 4; ++j) {
            uint32_t r[32];
            const uint32_t a = tmem + lane_off + kColO + 128 * c + 32 * j;
            tmem_ld32(a, r);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tmem_st32(a, r);
          }
          tmem_st_wait();
        } else {
          fail(B, p.status);  // carried to the next sub-tile's barrier
        }
      }
      // probabilities -> P (this thread's 32 tokens of its row): bf16 for
      // bf16 caches, fp16 for the dequantised 1-byte caches; l sums the
      // rounded values PV multiplies by.  P goes to shared memory (K-major,
      // 128-byte swizzle) once PV of sub-tile k - 2 has read the buffer.
      {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float pa_ = ex2_ftz(x[2 * i] - m_run), pb_ = ex2_ftz(x[2 * i + 1] - m_run);
          if constexpr (kByte) {
            const __half wa = __float2half_rn(pa_), wb = __float2half_rn(pb_);
            l_run += __half2float(wa) + __half2float(wb);
            pk[i] = uint32_t(__half_as_ushort(wa)) | (uint32_t(__half_as_ushort(wb)) << 16);
          } else {
            const __nv_bfloat16 wa = __float2bfloat16_rn(pa_), wb = __float2bfloat16_rn(pb_);
            l_run += __bfloat162float(wa) + __bfloat162float(wb);
            pk[i] = uint32_t(__bfloat16_as_ushort(wa)) | (uint32_t(__bfloat16_as_ushort(wb)) << 16);
          }
        }
        if constexpr (C::kPSmem) {
          const bool okp = k < 2 || mbar_wait(&B->pv_done[sb], ((k - 2) >> 1) & 1, abort_flag, kWaitLimitNs);
          if (!okp) fail(B, p.status);  // carried to the next sub-tile's barrier
          uint8_t* prow = smem + C::kOffP + sb * kPBytes + h * 128;
#pragma unroll
          for (int v = 0; v < 4; ++v)
            *reinterpret_cast<uint4*>(prow + (((4 * c + v) ^ (h & 7)) << 4)) =
                make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          fence_proxy_async_smem();
        } else {  // over the scores, which send() has read
          tmem_st16u(tmem + lane_off + kColS + sb * kSub + 16 * c, pk);
          tmem_st_wait();
          tc_fence_before();
        }
      }
      mbar_arrive(&B->p_full[sb]);
      if (s.last) {
        const bool ok2 = mbar_wait(&B->o_full, seg & 1, abort_flag, kWaitLimitNs);
        // the row's sum over both halves, added in a fixed order, through the
        // other parity's maxima (every thread read them before this
        // sub-tile's barrier; they are written again after the barrier below)
        float* rl = red + (sb ^ 1) * 256;
        rl[c * 128 + h] = l_run;
        if (soft_any(!ok2)) break;
        const float l_row = rl[h] + rl[128 + h];
        tc_fence_after();
        const float inv_l = l_row > 0.f ? __frcp_rn(l_row) : 0.f;  // 0: a row that saw no token
        float4* dst =
            reinterpret_cast<float4*>(p.partial_o + (size_t(s.seg) * p.heads + row) * kLatent + lat0 + 128 * c);
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_off + kColO + 128 * c + 32 * j, r);
          if (live) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[8 * j + i] = make_float4(__uint_as_float(r[4 * i]) * inv_l, __uint_as_float(r[4 * i + 1]) * inv_l,
                                           __uint_as_float(r[4 * i + 2]) * inv_l, __uint_as_float(r[4 * i + 3]) * inv_l);
          }
        }
        tc_fence_before();
        mbar_arrive(&B->o_free);
        if (rank == 0 && c == 0 && live)
          p.partial_lse[size_t(s.seg) * p.heads + row] = l_row > 0.f ? (m_run + log2f(l_row)) * kLn2 : -INFINITY;
        soft_sync();  // the sums are read before the next sub-tile writes its maxima there
        ++seg;
      }
      if (!C::kPSmem && have_next) {
        if (sn.first) load_q(sn);
        sent_ok = send(k + 1);
      }
      s = sn;
      have = have_next;
      ++k;
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
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  cluster_sync();  // the peer may still be sending into this CTA's shared memory until here
}

template <int kCode>
cudaError_t launch_hm(const DecodeParams& p, int clusters_per_group, cudaStream_t stream) {
  constexpr bool kByte = kCode != kCodeBf16;
  using C = HmCfg<kByte>;
  CUtensorMap ml, mr, mqr;
  const uint64_t rows = uint64_t(p.num_pages) * p.page_size, qrows = uint64_t(p.batch) * p.heads;
  const uint32_t box_rows = p.page_size < kSub ? p.page_size : kSub;
  const int eb = kByte ? 1 : 2;
  if (!make_map_2d(&ml, p.cache, eb, kRow, rows, 64, box_rows,
                   kByte ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_2d(&mr, p.cache, eb, kRow, rows, 32, box_rows,
                   kByte ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_map_2d(&mqr, p.q_full, 2, kRow, qrows, 32, kRowsG, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  static std::atomic<bool> attr[128];  // per device: attributes set (zero-initialised)
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 128 || !attr[dev]) {
    for (auto* k : {decode_hm_kernel<kCode, false, false>, decode_hm_kernel<kCode, true, false>,
                    decode_hm_kernel<kCode, false, true>, decode_hm_kernel<kCode, true, true>}) {
      const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(C::kSmem));
      if (e != cudaSuccess) return e;
    }
    if (dev >= 0 && dev < 128) attr[dev] = true;
  }
  const bool pad = p.heads % kRowsG != 0;
  auto* kernel = p.q_len > 1 ? (pad ? decode_hm_kernel<kCode, true, true> : decode_hm_kernel<kCode, true, false>)
                             : (pad ? decode_hm_kernel<kCode, false, true> : decode_hm_kernel<kCode, false, false>);
  return launch_pdl(kernel, dim3(2 * clusters_per_group * p.num_groups), dim3(C::kThreads), C::kSmem, stream, 2, ml,
                    mr, mqr, p);
}

template <int kCode>
int hm_capacity() {  // CTA pairs of this kernel that can be resident at once on this device
  using C = HmCfg<kCode != kCodeBf16>;
  static std::atomic<int> cached[128];  // per device (zero-initialised)
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 128 && cached[dev] > 0) return cached[dev];
  if (cudaFuncSetAttribute(decode_hm_kernel<kCode, false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(C::kSmem)) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, decode_hm_kernel<kCode, false, false>, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return 0;
  }
  if (dev >= 0 && dev < 128) cached[dev] = n;
  return n;
}

}  // namespace

int decode_rows128_capacity(int code) {
  return code == kCodeInt8 ? hm_capacity<kCodeInt8>() : code == kCodeE4m3 ? hm_capacity<kCodeE4m3>()
                                                                          : hm_capacity<kCodeBf16>();
}

cudaError_t launch_decode_rows128(const DecodeParams& p, int code, int clusters_per_group, cudaStream_t stream) {
  return code == kCodeInt8   ? launch_hm<kCodeInt8>(p, clusters_per_group, stream)
         : code == kCodeE4m3 ? launch_hm<kCodeE4m3>(p, clusters_per_group, stream)
                             : launch_hm<kCodeBf16>(p, clusters_per_group, stream);
}

}  // namespace mla
