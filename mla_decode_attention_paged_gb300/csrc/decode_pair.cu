// decode_pair.cu -- split-KV MLA decode attention for bf16 caches on CTA
// pairs (thread-block clusters of two), tcgen05 tensor cores fed by TMA.
//
// What it computes ("The Weight Absorption Trick"; "Seven Ways LLMs Handle
// Attention", section 5; "Flash-Decoding and FlashInfer"): for one head group
// of one sequence and one contiguous range of its tokens, with
// q_full[h] = [W^UK_h^T q_nope_h | q_pe_h] (576 wide) and the cached rows
// c_t = [latent | RoPE key] (576 wide),
//     s[t][h] = scale * q_full[h] . c_t
//     o_lat[h] = sum_t softmax(s[., h])_t * c_t[0:512]
// and emits o_lat (normalised within the range) with the range's lse.
//
// Why pairs.  Both products read the same cached tile (the latent part is
// K of QK^T and V of PV), so a tile must stay in shared memory from its QK^T
// until its PV, across the softmax in between.  A 128-token tile is 147 KB;
// one SM holds about 1.3 of them, which serialises load -> QK^T -> softmax ->
// PV.  Here the two CTAs of a cluster (two SMs) split every tile by columns:
// CTA r holds latent columns [256 r, 256 r + 256) and RoPE columns
// [512 + 32 r, 512 + 32 r + 32): 72 KB per tile, so each SM keeps two tiles
// in flight.
//   * QK^T: each CTA forms the partial scores over its columns, S_r^T
//     [128 tok x HC] = C_r [128 x 288] * Q_r^T, and sends them, in log2
//     units rounded to fp16, to the other CTA through distributed shared
//     memory (4 KB for 16 heads);
//   * both CTAs add the same two fp16 values (so both get the same bits),
//     run the same softmax and hold the same P^T;
//   * PV: each CTA accumulates its own 256 latent columns of O^T.
// Every page is read from HBM once for all heads of the group.
//
// Orientation as in the single-CTA kernel: the 128 tokens of a tile are the
// MMA's M extent and the heads its N extent:
//     S_r^T [128 x HC]   = C_r [128 x 288] * Q_r^T           (A K-major)
//     O_r^T [256 x HC]  += C_r^T [256 x 128] * P^T           (A MN-major)
//
// Warp roles (256 threads per CTA):
//   warp 0     TMA producer: Q of each segment and the first half of each
//              tile's latent boxes
//   warp 1     TMEM allocation; lane 0 issues the QK^T MMAs
//   warp 2     PV: lane 0 issues the MMAs; the warp clears the ragged tail
//              rows of a sequence's last tile first
//   warp 3     TMA producer: the second half of the latent boxes and the
//              RoPE columns
//   warps 4-7  exchange of partial scores, softmax (one thread per token
//              row), epilogue
// Every wait is bounded: on timeout the CTA records MLA_ERR_DEVICE_TIMEOUT,
// drains, frees its tensor memory and returns (the other CTA of its pair
// then times out on the exchange and does the same).
#include <atomic>
#include "blackwell_ptx.cuh"
#include "decode_common.cuh"
#include "params.cuh"

namespace mla {
namespace {

using namespace ptx;
using namespace dc;

constexpr int kPairThreads = 256;
constexpr uint32_t kBoxBytes = 16384;           // [128 tokens x 64 columns] bf16, 128-byte swizzle
constexpr uint32_t kPairBytes = 2 * kBoxBytes;  // 128 latent columns: one O^T chunk
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr float kRescaleThreshold = 8.f;          // log2 units
constexpr bool kPrefetchNext = true;              // L2 prefetch of the next tile's boxes
constexpr int kMaxSlots = 6;                      // barrier array size of each ring
constexpr int NC = 2;                             // CTAs per cluster

// HC heads per pair; CTA r of the pair holds latent columns [256 r, 256 r +
// 256) -- kChunks chunks of 128 -- and RoPE columns [512 + 32 r, + 32).
template <int HC>
struct PairCfg {
  static constexpr int kChunks = 4 / NC;            // 128-column latent chunks per CTA and tile
  static constexpr int kRopeCols = 64 / NC;         // RoPE columns per CTA (64-byte rows)
  static constexpr uint32_t kRopeBytes = kTile * kRopeCols * 2;
  static constexpr uint32_t kRopeSbo = 8 * kRopeCols * 2;  // 8-row swizzle atom
  static constexpr uint32_t kRopeSwizzle = kSwizzle64B;
  static constexpr int kNumPair = 4;                // chunk slots: two tiles (an even count keeps both
                                                    // producers, one chunk each, in step)
  static constexpr int kNumRope = 3;                // RoPE slots (one per tile)
  static constexpr int kBoxesPerProducer = 2;       // the two producers load one chunk (two boxes) each
  static constexpr uint32_t kQBytes = kChunks * 2 * HC * 128 + HC * kRopeCols * 2;
  static constexpr uint32_t kPBytes = kTile * HC * 2;  // P^T, bf16
  static constexpr uint32_t kXBytes = kTile * HC * 2;  // the other CTA's partial S^T, fp16
  static constexpr uint32_t kOffPair = 0;
  static constexpr uint32_t kOffRope = kOffPair + kNumPair * kPairBytes;
  static constexpr uint32_t kOffQ = kOffRope + ((kNumRope * kRopeBytes + 1023) & ~1023u);
  static constexpr uint32_t kOffQRope = kOffQ + kChunks * 2 * HC * 128;
  static constexpr uint32_t kOffP = kOffQ + ((kQBytes + 1023) & ~1023u);
  static constexpr uint32_t kOffX = kOffP + 2 * kPBytes;  // [2 buffers] of the peer's partials
  static constexpr uint32_t kOffMisc = kOffX + 2 * kXBytes;
  static constexpr uint32_t kMiscBytes = 2560;
  static constexpr uint32_t kSmem = kOffMisc + kMiscBytes + 1024;  // +1024: base alignment slack
  static constexpr uint32_t kColS = 0;                             // + buf * HC
  static constexpr uint32_t kColO = 2 * HC;                        // + c * HC
  static constexpr uint32_t kTmemCols = (2 + kChunks) * HC <= 64 ? 64 : ((2 + kChunks) * HC <= 128 ? 128 : 256);
  static_assert(kSmem <= 232448, "dynamic shared memory of one CTA");
  static_assert(kNumPair <= kMaxSlots && kNumRope <= kMaxSlots, "barrier arrays");
  static_assert(512 + 13 * HC * 4 <= kMiscBytes, "barriers, maxima, sums and reciprocal sums");
  static_assert(kOffQ % 1024 == 0 && kOffQRope % 256 == 0, "swizzle atoms");
};

struct PairBarriers {
  uint64_t full_pair[kMaxSlots], empty_pair[kMaxSlots], full_rope[kMaxSlots], empty_rope[kMaxSlots];
  uint64_t q_full, q_empty, s_full[2], x_full[2], p_full[2], pv_done[2], o_full, o_free, drain[2];
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void fail(PairBarriers* B, int* status) {
  B->abort = 1;
  set_status(status, MLA_ERR_DEVICE_TIMEOUT);
}

// kCausal: multi-token decode (q_len > 1) masks the scores of each row's
// later positions on a sequence's last tiles; single-token decode does not
// carry the per-tile check.
template <int HC, bool kCausal>
__global__ void __launch_bounds__(kPairThreads, 1)
    decode_pair_kernel(const __grid_constant__ CUtensorMap tmap_latent, const __grid_constant__ CUtensorMap tmap_rope,
                       const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_qrope,
                       DecodeParams p) {
  using C = PairCfg<HC>;
  extern __shared__ uint8_t smem_raw[];
  // the same offset in every CTA: the others' exchange buffers and barriers are found by mapa
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  PairBarriers* B = reinterpret_cast<PairBarriers*>(smem + C::kOffMisc);
  // [2][HC][4] maxima, [HC][4] sums of l, [HC] 1 / l
  float* red = reinterpret_cast<float*>(smem + C::kOffMisc + 512);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kNumPair; ++i) {
      mbar_init(&B->full_pair[i], 1);
      mbar_init(&B->empty_pair[i], 1);
    }
    for (int i = 0; i < C::kNumRope; ++i) {
      mbar_init(&B->full_rope[i], 1);
      mbar_init(&B->empty_rope[i], 1);
    }
    mbar_init(&B->q_full, 1);
    mbar_init(&B->q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&B->s_full[i], 1);
      mbar_init(&B->x_full[i], 1);  // armed by one local thread; the other CTAs' bytes complete it
      mbar_init(&B->p_full[i], 128);
      mbar_init(&B->pv_done[i], 1);
      mbar_init(&B->drain[i], 1);
    }
    mbar_init(&B->o_full, 1);
    mbar_init(&B->o_free, 128);
    B->abort = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmap_latent);
    prefetch_tensormap(&tmap_rope);
    prefetch_tensormap(&tmap_q);
    prefetch_tensormap(&tmap_qrope);
  }
  if (warp == 1) {
    tmem_alloc(&B->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  cluster_sync();  // every CTA's barriers exist before any sends to another
  tc_fence_after();
  const uint32_t tmem = B->tmem_base;
  griddep_wait();  // the plan and Q come from the kernel before
  griddep_launch_dependents();

  const int G = p.num_groups, clus = blockIdx.x / NC, g = clus % G, cp = clus / G, Cp = (gridDim.x / NC) / G;
  const long long S = p.status[1];  // effective split count from the plan
  const long long pa = (cp * S) / Cp, pb = ((cp + 1) * S) / Cp;
  const volatile int* abort_flag = &B->abort;
  const int P = p.page_size;
  const int lat0 = (kLatent / NC) * int(rank), rope0 = kLatent + C::kRopeCols * int(rank);  // this CTA's columns

  if ((warp == 0 || warp == 3) && lane == 0) {
    // ------------------------------------------------------------ producers
    // One thread cannot issue TMA copies fast enough for an SM's share of
    // HBM (about 0.15-0.2 us per 8 KB box), so two warps share the work:
    // warp 0 loads Q and the first half of every tile's latent boxes, warp 3
    // the second half and the RoPE columns.
    const int role = warp == 0 ? 0 : 1;
    TileWalkerT<true> walk;
    walk.init(p.tile_start, p.seg_base, p.len, p.batch, int(S), pa, pb);
    const uint32_t page_bytes = uint32_t(P) * 128, rope_page_bytes = uint32_t(P) * C::kRopeCols * 2;
    uint32_t pair_it = 0, rope_it = 0, seg = 0;
    TileInfo t, tn;
    // page ids two tiles ahead: tile k + 1's are in registers (and arrived)
    // when tile k starts, for the L2 prefetch; tile k + 2's are on their way
    TileWalkerT<true> look = walk;
    TilePages pages, next_pages, next2_pages;
    bool have_next = look.next(tn), have_next2 = false;
    if (have_next) next_pages.fetch(p, tn);
    if (have_next) {
      have_next2 = look.next(tn);
      if (have_next2) next2_pages.fetch(p, tn);
    }
    bool ok = true;
    while (ok && walk.next(t)) {
      pages = next_pages;
      next_pages = next2_pages;
      have_next = have_next2;
      have_next2 = have_next && look.next(tn);
      if (have_next2) next2_pages.fetch(p, tn);
      if (t.first && role == 0) {
        if (seg > 0 && !(ok = mbar_wait(&B->q_empty, (seg - 1) & 1, abort_flag, kWaitLimitNs))) break;
        mbar_arrive_expect_tx(&B->q_full, C::kQBytes);
        const int qrow = t.b * p.heads + g * HC;
        for (int j = 0; j < 2 * C::kChunks; ++j)
          tma_load_2d(smem + C::kOffQ + j * HC * 128, &tmap_q, lat0 + 64 * j, qrow, &B->q_full);
        tma_load_2d(smem + C::kOffQRope, &tmap_qrope, rope0, qrow, &B->q_full);
        ++seg;
      }
      const int npg = pages.npg;
      int rows[kTile / 16];
      pages.rows(p, rows);
      if (kPrefetchNext && have_next && G == 1) {
        // the next tile's boxes into L2 now: its copies, issued once a slot
        // frees, then find them there instead of waiting on DRAM (with
        // several head groups each tile is read by every group, and the
        // extra requests cost more than they save)
        int nrows[kTile / 16];
        next_pages.rows(p, nrows);
#pragma unroll 1
        for (int i = 0; i < next_pages.npg; ++i) {
          for (int b = 0; b < C::kBoxesPerProducer; ++b)
            tma_prefetch_2d(&tmap_latent, lat0 + 64 * (C::kBoxesPerProducer * role + b), nrows[i]);
          if (role == 1) tma_prefetch_2d(&tmap_rope, rope0, nrows[i]);
        }
      }
      {
        // producer `role` loads chunk `role` of this CTA's two (its two 64-column boxes)
        const int c = role, b0 = 0;
        const uint32_t it = pair_it + c;
        const uint32_t slot = it % C::kNumPair;
        if (!(ok = mbar_wait(&B->empty_pair[slot], ((it / C::kNumPair) & 1) ^ 1, abort_flag, kWaitLimitNs))) break;
        uint8_t* dst = smem + C::kOffPair + slot * kPairBytes;
        mbar_arrive_expect_tx(&B->full_pair[slot], C::kBoxesPerProducer * npg * page_bytes +
                                                       (p.inject_wait_timeout && it == 0 ? 16 : 0));
#pragma unroll 1
        for (int i = 0; i < npg; ++i)
          for (int b = b0; b < b0 + C::kBoxesPerProducer; ++b)
            tma_load_2d(dst + b * kBoxBytes + i * page_bytes, &tmap_latent, lat0 + 128 * c + 64 * b, rows[i],
                        &B->full_pair[slot]);
      }
      pair_it += C::kChunks;
      if (role == 0) continue;
      const uint32_t slot = rope_it % C::kNumRope;
      if (!(ok = mbar_wait(&B->empty_rope[slot], ((rope_it / C::kNumRope) & 1) ^ 1, abort_flag, kWaitLimitNs)))
        break;
      uint8_t* dst = smem + C::kOffRope + slot * C::kRopeBytes;
      mbar_arrive_expect_tx(&B->full_rope[slot], npg * rope_page_bytes);
#pragma unroll 1
      for (int i = 0; i < npg; ++i) tma_load_2d(dst + i * rope_page_bytes, &tmap_rope, rope0, rows[i], &B->full_rope[slot]);
      ++rope_it;
    }
    if (!ok) fail(B, p.status);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ QK issuer
    // S_r^T[k & 1] = C_r * Q_r^T: this CTA's latent chunks (8 MMAs each) and
    // its RoPE columns (one MMA per 16).  Before overwriting S^T[k & 1] it waits for the softmax of
    // tile k - 2 (which read it) to finish.
    TileWalkerT<true> walk;
    walk.init(p.tile_start, p.seg_base, p.len, p.batch, int(S), pa, pb);
    constexpr uint32_t id_qk = idesc_f32acc(128, HC, false, false, false);
    constexpr uint64_t kDescK = smem_desc(0, 16, 1024, kSwizzle128B);   // K-major, 128-byte swizzle
    constexpr uint64_t kDescRope = smem_desc(0, 16, C::kRopeSbo, C::kRopeSwizzle);  // K-major, narrow rows
    uint32_t k = 0, seg = 0, pair_it = 0;
    TileInfo t;
    bool ok = true;
    while (ok && walk.next(t)) {
      if (k >= 2 && !(ok = mbar_wait(&B->p_full[k & 1], ((k - 2) >> 1) & 1, abort_flag, kWaitLimitNs))) break;
      if (t.first && !(ok = mbar_wait(&B->q_full, seg & 1, abort_flag, kWaitLimitNs))) break;
      const uint32_t d_s = tmem + C::kColS + (k & 1) * HC;
      for (int c = 0; c < C::kChunks; ++c, ++pair_it) {
        const uint32_t slot = pair_it % C::kNumPair;
        if (!(ok = mbar_wait(&B->full_pair[slot], (pair_it / C::kNumPair) & 1, abort_flag, kWaitLimitNs))) break;
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
      {
        const uint64_t a0 = kDescRope | desc_addr(sbase + C::kOffRope + rslot * C::kRopeBytes);
        const uint64_t b0 = kDescRope | desc_addr(sbase + C::kOffQRope);
#pragma unroll
        for (int kk = 0; kk < C::kRopeCols / 16; ++kk) mma_bf16(d_s, a0 + 2 * kk, b0 + 2 * kk, id_qk, 1);
      }
      mma_commit(&B->s_full[k & 1]);
      mma_commit(&B->empty_rope[rslot]);
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
    // O_r^T[c] (+)= C_r^T[128c .. 128c + 128) * P^T once the softmax of the
    // tile is done; each pair slot is released as soon as its MMAs complete.
    TileWalkerT<true> walk;
    walk.init(p.tile_start, p.seg_base, p.len, p.batch, int(S), pa, pb);
    constexpr uint32_t id_pv = idesc_f32acc(128, HC, true, true, false);
    constexpr uint64_t kDescMN = smem_desc(0, kBoxBytes, 1024, kSwizzle128B);  // MN-major, 128-byte swizzle
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
      for (int c = 0; c < C::kChunks; ++c, ++pair_it) {
        const uint32_t slot = pair_it % C::kNumPair;
        if (tail_rows) {
          // they meet zero weights in P^T but must be finite: clear them (rows
          // past the loaded pages hold whatever the slot held before)
          uint8_t* base = smem + C::kOffPair + slot * kPairBytes;
          for (int i = lane; i < tail_rows * 16; i += 32)
            *reinterpret_cast<uint4*>(base + ((i >> 3) & 1) * kBoxBytes + (t.valid + (i >> 4)) * 128 + (i & 7) * 16) =
                make_uint4(0, 0, 0, 0);
          fence_proxy_async_smem();
          __syncwarp();
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
  } else if (warp >= 4) {
    // ------------------------------------------------------------ exchange / softmax / epilogue
    const int q4 = warp - 4, st = threadIdx.x - 128;  // st = token row of S^T = TMEM lane
    const uint32_t lane_off = uint32_t(q4 * 32) << 16;
    // this thread's row of an exchange buffer; 16-byte pieces rotated by row to spread banks
    constexpr int kV4 = HC / 8;
    const uint32_t x_local = sbase + C::kOffX + st * HC * 2;
    TileWalkerT<true> walk;
    walk.init(p.tile_start, p.seg_base, p.len, p.batch, int(S), pa, pb);
    float m_run[HC], l_run[HC];
    uint32_t tile_i = 0, seg = 0;
    TileInfo t;
    while (walk.next(t)) {
      const uint32_t buf = tile_i & 1;
      const bool valid = st < t.valid;
      // S_r^T of this tile; and PV of tile k - 2, which read the P^T buffer
      // this tile writes, must be complete
      bool ok = mbar_wait(&B->s_full[buf], (tile_i >> 1) & 1, abort_flag, kWaitLimitNs);
      tc_fence_after();
      float x[HC];
      if (ok) {
        // this CTA's partial scores in log2 units, rounded to fp16: the
        // exchange sends fp16 (distributed shared memory moves only ~12-15
        // GB/s per SM here) and both CTAs add the same two fp16 values, so
        // both get the same bits
        uint32_t hx[HC / 2];
#pragma unroll
        for (int h0 = 0; h0 < HC; h0 += 16) {
          float v[16];
          tmem_ld16(tmem + lane_off + C::kColS + buf * HC + h0, v);
#pragma unroll
          for (int i = 0; i < 8; ++i) hx[h0 / 2 + i] = pack_f16x2_sat(v[2 * i] * p.scale_log2, v[2 * i + 1] * p.scale_log2);
        }
        // partial scores to the peer CTA, into its buffer `buf`
        {
          const uint32_t peer = rank ^ 1u;
          const uint32_t rbar = mapa_shared(smem_u32(&B->x_full[buf]), peer);
          const uint32_t xr = mapa_shared(x_local + buf * C::kXBytes, peer);
#pragma unroll
          for (int v = 0; v < kV4; ++v)
            st_async_v4_b32(xr + (v ^ (st % kV4)) * 16, hx[4 * v], hx[4 * v + 1], hx[4 * v + 2], hx[4 * v + 3], rbar);
        }
        if (st == 0) mbar_arrive_expect_tx(&B->x_full[buf], C::kXBytes);
        ok = mbar_wait_cluster(&B->x_full[buf], (tile_i >> 1) & 1, abort_flag, kWaitLimitNs);
        if (ok) {
          // S = S_0 + S_1 (addition is commutative: both CTAs get the same bits)
#pragma unroll
          for (int v = 0; v < kV4; ++v) {
            const uint4 y = *reinterpret_cast<const uint4*>(smem + C::kOffX + buf * C::kXBytes + st * HC * 2 +
                                                            (v ^ (st % kV4)) * 16);
            const uint32_t yy[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 a = unpack_f16x2(hx[4 * v + i]), b = unpack_f16x2(yy[i]);
              x[8 * v + 2 * i] = a.x + b.x;
              x[8 * v + 2 * i + 1] = a.y + b.y;
            }
          }
        }
      }
#pragma unroll
      for (int h = 0; h < HC; ++h) x[h] = valid ? x[h] : -INFINITY;
      if (kCausal && causal_tile(p, t, walk.len_b)) causal_mask<HC>(x, p, g, walk.len_b, t.tile * kTile + st);
      // Running max: it only has to bound the scores to within
      // kRescaleThreshold (log2 units).  The first tile of a segment, and a
      // tile that breaks the bound, take the exact path (per-head tile max and,
      // where it moved, a rescale of O^T and l); otherwise one vote suffices.
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
            alpha[h] = 1.f;
          } else if (mt > m_run[h] + kRescaleThreshold) {
            alpha[h] = exp2f(m_run[h] - mt);
            m_run[h] = mt;
            l_run[h] *= alpha[h];
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
        for (int c = 0; c < C::kChunks; ++c)
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
      // PV of tile k - 2, which read the P^T buffer this tile writes, must be complete
      if (tile_i >= 2 && bar_any(!mbar_wait(&B->pv_done[buf], ((tile_i - 2) >> 1) & 1, abort_flag, kWaitLimitNs)))
        break;
      // probabilities -> P^T (bf16, MN-major, no swizzle: 8x8 core matrices)
      uint8_t* pt = smem + C::kOffP + buf * C::kPBytes;
#pragma unroll
      for (int h0 = 0; h0 < HC; h0 += 8) {
        uint32_t packed[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int ha = h0 + 2 * i, hb = ha + 1;
          const __nv_bfloat16 wa = __float2bfloat16_rn(ex2_ftz(x[ha] - m_run[ha]));
          const __nv_bfloat16 wb = __float2bfloat16_rn(ex2_ftz(x[hb] - m_run[hb]));
          l_run[ha] += __bfloat162float(wa);
          l_run[hb] += __bfloat162float(wb);
          packed[i] = uint32_t(__bfloat16_as_ushort(wa)) | (uint32_t(__bfloat16_as_ushort(wb)) << 16);
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
        float* rl = red + 8 * HC;  // [HC][4] sums of l
        {
          float tmp[HC];
#pragma unroll
          for (int h = 0; h < HC; ++h) tmp[h] = l_run[h];
          const float ls = warp_transpose_reduce<HC, false>(tmp, lane);
          if (HC == 32 || !(lane & 1)) rl[(HC == 32 ? lane : lane >> 1) * 4 + q4] = ls;
        }
        if (bar_any(!ok2)) break;
        // thread h computes head h's 1 / l once: sixteen or thirty-two IEEE
        // reciprocals in a row in every thread took ~1.3 us, at every
        // segment end, with the pipeline stalled behind it
        float* rinv = red + 12 * HC;  // [HC]
        float ih = 0.f;
        if (st < HC) {
          const float4 l4 = reinterpret_cast<const float4*>(rl)[st];
          const float l = (l4.x + l4.y) + (l4.z + l4.w);
          ih = l > 0.f ? __frcp_rn(l) : 0.f;  // 0: a row with no visible token (multi-token decode)
          rinv[st] = ih;
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
        float* dst = p.partial_o + (size_t(t.seg) * p.heads + g * HC) * kLatent + lat0;
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
#pragma unroll
          for (int h0 = 0; h0 < HC; h0 += 16) {
            float v[16];
            tmem_ld16(tmem + lane_off + C::kColO + c * HC + h0, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) dst[(h0 + i) * kLatent + c * 128 + st] = v[i] * inv_l[h0 + i];
          }
        tc_fence_before();
        mbar_arrive(&B->o_free);
        if (rank == 0 && st < HC) {  // thread h writes head h's lse
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
  cluster_sync();  // other CTAs may still be sending into this CTA's shared memory until here
}

template <int HC>
cudaError_t launch_pair(const DecodeParams& p, int clusters_per_group, cudaStream_t stream) {
  using C = PairCfg<HC>;
  CUtensorMap ml, mr, mq, mqr;
  const uint64_t rows = uint64_t(p.num_pages) * p.page_size, qrows = uint64_t(p.batch) * p.heads;
  if (!make_map_2d(&ml, p.cache, 2, kRow, rows, 64, p.page_size, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_2d(&mr, p.cache, 2, kRow, rows, C::kRopeCols, p.page_size, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_map_2d(&mq, p.q_full, 2, kRow, qrows, 64, HC, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_2d(&mqr, p.q_full, 2, kRow, qrows, C::kRopeCols, HC, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  static std::atomic<bool> attr[128];  // per device: attributes set (zero-initialised)
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 128 || !attr[dev]) {
    for (auto* k : {decode_pair_kernel<HC, false>, decode_pair_kernel<HC, true>}) {
      const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(C::kSmem));
      if (e != cudaSuccess) return e;
    }
    if (dev >= 0 && dev < 128) attr[dev] = true;
  }
  auto* kernel = p.q_len > 1 ? decode_pair_kernel<HC, true> : decode_pair_kernel<HC, false>;
  return launch_pdl(kernel, dim3(NC * clusters_per_group * p.num_groups), dim3(kPairThreads), C::kSmem, stream, NC,
                    ml, mr, mq, mqr, p);
}

template <int HC>
int max_clusters() {  // CTA pairs that can be resident at once on this device
  static std::atomic<int> cached[128];  // per device (zero-initialised)
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 128 && cached[dev] > 0) return cached[dev];
  if (cudaFuncSetAttribute(decode_pair_kernel<HC, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(PairCfg<HC>::kSmem)) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(NC);
  cfg.blockDim = dim3(kPairThreads);
  cfg.dynamicSmemBytes = PairCfg<HC>::kSmem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = NC;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, decode_pair_kernel<HC, false>, &cfg) != cudaSuccess || n <= 0) return 0;
  if (dev >= 0 && dev < 128) cached[dev] = n;
  return n;
}

}  // namespace

int decode_pair_capacity(int hc) { return hc == 16 ? max_clusters<16>() : max_clusters<32>(); }

cudaError_t launch_decode_pair(const DecodeParams& p, int hc, int clusters_per_group, cudaStream_t stream) {
  return hc == 16 ? launch_pair<16>(p, clusters_per_group, stream) : launch_pair<32>(p, clusters_per_group, stream);
}

}  // namespace mla
