// Absorbed-MLA latent attention on 5th-generation tensor cores (sm_103a).
//
// "Mla Analysis" skill page, "Absorption Trick (FlashMLA)": with the key and
// value up-projections folded out, attention runs entirely in the latent
// space: scores = Qz Z^T (+ the decoupled RoPE part q_pe K_pe^T, "Tensor
// Shapes": K_pe [B,T,P] shared by all heads) and O_lat = softmax(scores) Z.
// The same latent row Z_m serves as key and as value, and every query row of
// a sequence (h heads x s new tokens) reads the same Z, which is what makes
// the form compute-heavy ("Cost Models", FlashMLA: AI ~ 228 FLOP/B at s = 1).
//
// Kernel design: a cluster of two CTAs per (sequence, context chunk, 128-row
// tile of the packed h*s query rows, row = head*s + token), one per SM.
//   * Tensor Memory (128 lanes x 512 fp32 columns per SM) holds exactly the
//     fp32 O_lat of 128 rows x k = 512, so the work is split by role instead of
//     by output columns (which would make both CTAs compute the same scores):
//       - the S CTA (cluster rank 0) keeps Qz of its 128 rows in Tensor Memory
//         (256 columns, the A operand) and q_pe in shared memory, and computes
//         S = Qz Z^T + q_pe K_pe^T one 128-key tile (two pages) at a time into
//         two 128-column S buffers (tcgen05.mma kind::f16, M=128 N=128, B = the
//         cache chunks in shared memory); eight softmax warps (thread = row, each
//         warp half of a tile's keys, row maxima exchanged through shared memory)
//         turn S into P (bf16) and ship it with the row rescale factors to the O
//         CTA's shared memory in one bulk copy per tile (cp.async.bulk
//         shared::cta -> shared::cluster, completing on the O CTA's mbarrier);
//       - the O CTA (rank 1) keeps the whole fp32 O_lat [128 x 512] in Tensor
//         Memory and accumulates O += P Z (M=128 N=256 K=16, A = P and B = the
//         Z slab, both in shared memory), streaming Z itself; its MMA commits
//         free the P buffers of the S CTA (a commit multicast to its mbarrier).
//     Every cache byte enters each SM's shared memory once per tile, and the
//     scores are computed once ("Cost Models", FlashMLA FLOP count).
//   * The query tile reaches Tensor Memory through the S ring's first lap: TMA
//     boxes of [128 rows x 64] land in the ring slots and the softmax warps move
//     them (shared -> registers -> tcgen05.st) before the slots carry cache.
//   * Cache chunks are [128 keys x 64 dims], two TMA boxes of one 64-token
//     page each (128-byte swizzle); the O ring carries [64 keys x 256 columns].
//   * Online softmax with a lazily moved reference maximum: a row's reference
//     moves only when its maximum grows past it by 2^8 (P stays below 256); the
//     O CTA then rescales those rows of O in Tensor Memory before the tile's
//     MMAs (rare after the first tile). Exponentials use ex2.approx.
//   * Keys past a row's causal limit (token i of s sees keys 0 .. L - s + i)
//     are masked in the softmax; Z rows past the sequence end are zeroed in
//     shared memory before the O MMAs (a cache may hold anything there), and
//     the second page of a last tile that lies wholly past the end is skipped.
//   * Output: with one chunk, bf16 O_lat and the LSE directly; otherwise fp32
//     partials (O / l, LSE) merged by the combine kernel. The S CTA writes the
//     LSE, the O CTA the rows (staged through shared memory, whole row segments).
//   * Every mbarrier wait is bounded; a CTA whose wait runs out records the
//     error, raises its own and its peer's abort flag, stops issuing, waits for
//     its own copies and MMAs and leaves through the final cluster barrier.
//   * Launched as a programmatic dependent of the previous kernel on the
//     stream: barrier set-up, Tensor Memory allocation, the cluster barrier and
//     the tensor-map prefetch run before griddepcontrol.wait, every global read
//     after it.
#include <cuda.h>

#include <climits>

#include "common.cuh"
#include "internal.h"

namespace decattn {

namespace {

constexpr int TK = 128;                    // keys per tile (two 64-token pages)
constexpr int HK = 64;                     // keys per page / per TMA box / per softmax warp
constexpr int BM = 128;                    // query rows per row tile (MMA M)
constexpr int NSB = 2;                     // S buffers in Tensor Memory (S CTA)
constexpr int NMSG = 2;                    // P message buffers (staging in S, landing in O)
constexpr int NSMW = 8;                    // softmax warps (S) / rescale + epilogue warps (O)
constexpr int NTHREADS = 32 * (2 + NSMW);  // producer, MMA issuer, NSMW row warps
constexpr int HALF_BOX = HK * 128;         // one [64 keys x 64 dims] box, 128-byte rows
constexpr int CHUNK = TK * 128;            // one [128 keys x 64 dims] chunk (two boxes)
constexpr int P_BLK = BM * HK * 2;         // P [128 rows x 64 keys] bf16, K-major, 128-byte swizzle
constexpr int MSG_ALPHA = 2 * P_BLK;       // [128] float row rescale factors
constexpr int MSG_FLAGS = MSG_ALPHA + BM * 4;  // [4] per-quadrant "a row was rescaled" words
constexpr int MSG_BYTES = MSG_FLAGS + 16;
constexpr int MSG_STRIDE = 34 * 1024;      // 1024-byte aligned message slots
constexpr uint32_t kMsgPiece = ((MSG_BYTES + 15) / 16 + 15) & ~15u;  // one of 16 pieces of a message copy
constexpr int FIN_BYTES = BM * 4;          // [128] float 1/l, sent once at the end
constexpr int S_NR = 5;                    // S-ring slots (CPI chunks each)
constexpr int O_NR = 4;                    // O-ring slots
constexpr int SB0 = 256;                   // first S buffer column (Qz holds columns 0 .. k/2-1)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.f;                        // move the reference max only past 2^8
constexpr unsigned long long kTeardownNs = 1000000000ull;  // 1 s for own copies / MMAs at exit
constexpr unsigned long long kTestWaitNs = 1000000ull;     // 1 ms forced-timeout wait
constexpr uint32_t kRankS = 0, kRankO = 1;
constexpr int kBarA = 1, kBarB = 2;        // named barriers of the row warps

static_assert(MSG_BYTES % 16 == 0 && MSG_BYTES <= MSG_STRIDE && kMsgPiece % 16 == 0, "message");
static_assert(SB0 + NSB * TK <= 512, "tensor memory");

constexpr int cmax(int a, int b) { return a > b ? a : b; }

template <int KL, int P>
struct MlaCfg {
  static constexpr int NBL = KL / 64;                   // latent chunks per tile (= query boxes)
  static constexpr int NCH = NBL + 1;                   // + the RoPE chunk
  // chunks per S-ring item: two, in five 32 KB slots. Each wait / commit of the ring costs
  // ~250 cycles of the issuing warp, but finer items keep more of the ring in flight:
  // against three chunks in three slots this measured 52.9 vs 53.5 us at s = 1 and 268
  // vs 269 us at s = 8 (s = 4, 32 and 64 lose 1.5-4 %), and one 80 KB item of five
  // chunks in two slots 55.4 / 295 us. At k = 512 the RoPE chunk forms the tile's last
  // item on its own.
  static constexpr int CPI = 2;
  static constexpr int NITEM = (NCH + CPI - 1) / CPI;   // S-ring items per tile
  static constexpr int S_ITEM = CPI * CHUNK;
  static constexpr int QS = (NBL + CPI - 1) / CPI;      // ring slots of the query lap
  static constexpr int LAT0 = NBL < CPI ? NBL : CPI;    // latent chunks of a full S-ring item
  static constexpr int LATL = NBL - (NITEM - 1) * CPI;  // latent chunks of a tile's last item (+ RoPE; may be 0)
  static constexpr int PE_ROW = P * 2;                  // bytes per RoPE row
  static constexpr uint32_t PE_SWZ = PE_ROW == 128 ? kSw128 : (PE_ROW == 64 ? kSw64 : kSw32);
  static constexpr int PE_HALF = HK * PE_ROW;           // one RoPE box (64 keys)
  static constexpr int ON = KL < 256 ? KL : 256;        // O MMA N (columns per O-ring item)
  static constexpr int NH = KL / ON;                    // O column blocks
  static constexpr int O_ITEM = HK * ON * 2;            // [64 keys x ON columns]
  static constexpr int OCOLS = KL / 2;                  // O columns per row warp (rescale, epilogue)
  // S CTA: one P staging slot, q_pe, the S-ring
  static constexpr int OFF_STG = 0;
  static constexpr int OFF_QPE = MSG_STRIDE;
  static constexpr int OFF_SRING = OFF_QPE + ((BM * PE_ROW + 1023) & ~1023);
  // O CTA: NMSG message slots (written by the S CTA's copies), the O-ring
  static constexpr int OFF_MSG = 0;
  static constexpr int OFF_ORING = NMSG * MSG_STRIDE;
  // both: 1/l, the row-statistics exchange and the barriers at the same offsets (peer-addressed)
  static constexpr int OFF_FIN = cmax(OFF_SRING + S_NR * S_ITEM, OFF_ORING + O_NR * O_ITEM);
  static constexpr int OFF_RED = OFF_FIN + FIN_BYTES;   // row maxima [2][2][128], row sums [2][128]
  static constexpr int OFF_BAR = OFF_RED + 6 * BM * 4;  // same offset in both CTAs
  static constexpr int SMEM = OFF_BAR + 512;
  static_assert(KL % 64 == 0 && KL / 2 <= SB0 && KL % ON == 0 && ON % 16 == 0 && ON <= 256, "latent width");
  static_assert(2 * CPI <= 16 && QS <= S_NR && LATL >= 0, "S-ring items");
  static_assert(P % 16 == 0 && PE_ROW <= 128, "rope width");
  static_assert(OCOLS % 32 == 0 && (OCOLS / 8 <= 32) && 32 % (OCOLS / 8) == 0, "row-warp columns");
  static_assert(NSMW * 32 * OCOLS * 2 <= O_NR * O_ITEM, "epilogue staging");
  static_assert(OFF_SRING % 1024 == 0 && OFF_ORING % 1024 == 0 && O_ITEM % 1024 == 0 && OFF_QPE % 1024 == 0,
                "swizzle alignment");
  static_assert(SMEM <= 232448, "shared memory");
};

// barrier slots (8 bytes each) at OFF_BAR, the same in both CTAs
enum : int {
  B_FULL = 0,       // [8] ring item landed
  B_EMPTY = 8,      // [8] ring item consumed
  B_SFULL = 16,     // [NSB] S tile in Tensor Memory (S CTA)
  B_SEMPTY = 18,    // [NSB] S tile read by the softmax warps (S CTA)
  B_PFULL = 20,     // [NMSG] P message landed (O CTA; the S CTA's copy completes on it)
  B_PFREE = 22,     // [NMSG] O CTA's MMAs done with message buffer (S CTA; O's commit arrives)
  B_QREADY = 24,    // Qz in Tensor Memory (S CTA)
  B_QPE = 25,       // q_pe landed (S CTA)
  B_FINFULL = 26,   // 1/l landed (O CTA)
  B_ODONE = 27,     // every O MMA issued before a rescale complete (O CTA)
  B_OFINAL = 28,    // every O MMA complete (O CTA)
  B_CREQ = 29,      // rescale request (or end marker) for the row warps (O CTA)
  B_CDONE = 30,     // rescale done (O CTA)
  B_TEST = 31,      // never signalled: the forced-timeout test waits on it
  B_FIN = 32,       // teardown: every tcgen05 op of the MMA issuer complete
  B_COUNT = 33
};
static_assert(S_NR <= 8 && O_NR <= 8, "ring barrier slots");

struct MlaParams {
  __nv_bfloat16* ws_ob;  // bf16 O / l partials [b*h*s, nsplit, k]
  const int32_t* seqlens;
  const int32_t* block_table;
  int max_pages, paged, capacity, num_pages;
  int b, s, h, rows, nsplit, chunk;
  int mtiles;                             // 128-row tiles per sequence
  int tail_whole, tail_k, tail_chunk;     // tail split (tail_k > 0), see the kernel
  float scale_log2;
  __nv_bfloat16* o_lat;
  float* lse;
  float* ws_lse;
  unsigned* err;
  unsigned long long wait_ns;
  int test_timeout;
};

// cache row of `key` of sequence bi (paged: through the block table; a 64-key box never
// crosses a page because boxes and pages are both 64 keys and chunks are whole tiles)
__device__ __forceinline__ int cache_row(const MlaParams& p, int bi, int key) {
  if (p.paged) {
    int page = p.block_table[(size_t)bi * p.max_pages + key / 64];
    if (page < 0 || page >= p.num_pages) {
      raise_error(p.err, kErrBadPage);
      page = 0;  // stay inside the pool; the result is flagged invalid
    }
    return page * 64 + (key % 64);
  }
  return bi * p.capacity + key;
}

// warp-uniform bounded wait (every lane polls; all agree on the outcome)
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns, volatile int* abort_flag) {
  if (__all_sync(0xffffffffu, mbar_test(bar, parity))) return true;
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, limit_ns, abort_flag));
}

// position in a ring: next slot and the phase parity of its current use
template <int NR>
struct RingPos {
  int slot = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void advance() {
    if (++slot == NR) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

// Tensor maps (all bf16, 128-byte swizzle):
//   tm_q3   Qz viewed as {64 columns, rows, k/64 chunks} (strides: row k*2 B, chunk 128 B),
//           box {64, 128, LAT0}: one box per query-lap slot, chunk-major as the MMAs read it
//   tm_qpe  q_pe [rows, p], box [128 rows, p]
//   tm_za / tm_zb   contiguous cache: Z viewed like Qz, boxes {64, 128, LAT0} / {64, 128, LATL}
//           (one box per S-ring item; tm_zb unused when the last item is the RoPE chunk
//           alone); paged pool: Z [rows, k] with boxes [64 rows, 64] (one
//           box per chunk and page), tm_zb unused
//   tm_kpe  K_pe [rows, p], box [128 rows, p] (contiguous) or [64 rows, p] (paged)
//   tm_zo   Z viewed like Qz, box {64, 64, ON/64}: one [64 keys x ON columns] O-ring item
// TMA serves about one box per few hundred cycles per SM (a single issuing thread half that),
// whatever its size up to tens of KB, so the cache streams use the largest boxes the layout
// allows.
template <int KL, int P, bool PAGED>
__global__ void __launch_bounds__(NTHREADS, 1)
    mla_pair_kernel(const __grid_constant__ CUtensorMap tm_q3, const __grid_constant__ CUtensorMap tm_qpe,
                    const __grid_constant__ CUtensorMap tm_za, const __grid_constant__ CUtensorMap tm_zb,
                    const __grid_constant__ CUtensorMap tm_kpe, const __grid_constant__ CUtensorMap tm_zo,
                    MlaParams p) {
  using C = MlaCfg<KL, P>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sb = smem_u32(smem);
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // This cluster's work: row tile mt of sequence bi over keys [kstart, kstart + chunk).
  //  * Fixed chunks: grid (2 * mtiles, nsplit, b).
  //  * Tail split (a 1-D grid): the units u = bi * mtiles + mt that fill whole waves of
  //    clusters run whole (u < tail_whole); each unit of the last, partial wave is cut into
  //    tail_k chunks of tail_chunk keys, so that wave takes 1 / tail_k of the time.
  // Partials go to record row (part_row0 + r) * part_n + split.
  int mt, split, bi, chunk, part_n;
  bool whole;
  size_t part_row0;
  if (p.tail_k > 0) {
    const int c = blockIdx.x >> 1;
    int u;
    if (c < p.tail_whole) {
      u = c;
      split = 0;
      whole = true;
      chunk = INT_MAX;
    } else {
      u = p.tail_whole + (c - p.tail_whole) / p.tail_k;
      split = (c - p.tail_whole) % p.tail_k;
      whole = false;
      chunk = p.tail_chunk;
    }
    bi = u / p.mtiles;
    mt = u % p.mtiles;
    part_n = p.tail_k;
    part_row0 = (size_t)(u - p.tail_whole) * BM;
  } else {
    mt = blockIdx.x >> 1;
    split = blockIdx.y;
    bi = blockIdx.z;
    chunk = p.chunk;
    whole = p.nsplit == 1;
    part_n = p.nsplit;
    part_row0 = (size_t)bi * p.rows + mt * BM;
  }
  const int kstart = split * chunk;
  const int qrow0 = bi * p.rows + mt * BM;  // first flattened [b*h*s] query row of the tile

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + B_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + B_COUNT) + 1;
  volatile int* req_tile = reinterpret_cast<volatile int*>(bars + B_COUNT) + 2;
  auto msg = [&](int m) { return smem + C::OFF_MSG + m * MSG_STRIDE; };

  // ---- set-up that touches no global memory (overlaps the previous kernel's end)
  if (threadIdx.x == 0) {
    for (int i = 0; i < 8; ++i) {
      mbar_init(&bars[B_FULL + i], 1);
      mbar_init(&bars[B_EMPTY + i], 1);
    }
    for (int i = 0; i < NSB; ++i) {
      mbar_init(&bars[B_SFULL + i], 1);
      mbar_init(&bars[B_SEMPTY + i], NSMW);
    }
    for (int i = 0; i < NMSG; ++i) {
      mbar_init(&bars[B_PFULL + i], 1);
      mbar_init(&bars[B_PFREE + i], 1);
    }
    mbar_init(&bars[B_QREADY], 1);
    mbar_init(&bars[B_QPE], 1);
    mbar_init(&bars[B_FINFULL], 1);
    mbar_init(&bars[B_ODONE], 1);
    mbar_init(&bars[B_OFINAL], 1);
    mbar_init(&bars[B_CREQ], 1);
    mbar_init(&bars[B_CDONE], NSMW);
    mbar_init(&bars[B_TEST], 1);
    mbar_init(&bars[B_FIN], 1);
    *abort_flag = 0;
    *req_tile = 0;
    // the one arrival of the final 1/l message's barrier, with its byte count (O CTA)
    if (rank == kRankO) mbar_expect_tx(&bars[B_FINFULL], FIN_BYTES);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_q3);
    prefetch_tmap(&tm_qpe);
    prefetch_tmap(&tm_za);
    prefetch_tmap(&tm_zb);
    prefetch_tmap(&tm_kpe);
    prefetch_tmap(&tm_zo);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // the peer's barriers exist before any copy, commit or store targets them

  // Each CTA allocates all 512 columns (one CTA per SM), so the allocation starts at
  // column 0; the kernel uses that address as a constant and checks it. A CTA that
  // cannot run (misaligned shared memory, unexpected allocation) aborts its pair.
  const bool setup_ok = ((sb & 1023u) == 0) && (*tmem_slot == 0);
  auto fail = [&]() {
    raise_error(p.err, kErrWaitTimeout);
    *abort_flag = 1;
    st_cluster_u32(mapa_shared(smem_u32((const void*)abort_flag), peer), 1u);
  };
  if (!setup_ok && threadIdx.x == 0) {
    raise_error(p.err, kErrLaunch);
    *abort_flag = 1;
    st_cluster_u32(mapa_shared(smem_u32((const void*)abort_flag), peer), 1u);
  }
  __syncthreads();

  // ---- inputs written by earlier kernels (queries, cache, lengths) are read from here on
  pdl_wait();
  pdl_trigger();
  const int L = p.seqlens[bi];
  const bool active = kstart < L && setup_ok && !*abort_flag;
  if (L <= 0 && whole) {  // empty sequence without a combine pass
    for (int idx = threadIdx.x; idx < BM * (KL / 8); idx += NTHREADS) {
      const int r = idx / (KL / 8);
      if (mt * BM + r >= p.rows) continue;
      const size_t grow = (size_t)qrow0 + r;
      if (rank == kRankO)
        *reinterpret_cast<uint4*>(p.o_lat + grow * KL + (idx % (KL / 8)) * 8) = make_uint4(0, 0, 0, 0);
      else if (p.lse && idx % (KL / 8) == 0)
        p.lse[grow] = -INFINITY;
    }
  }
  const int kend = chunk > L - kstart ? L : kstart + chunk;
  const int ntiles = active ? (kend - kstart + TK - 1) / TK : 0;
  constexpr uint32_t tmem = 0;

  if (rank == kRankS) {
    // =====================================================================================
    // S CTA
    if (warp == 0) {
      // ------------------------------------------------ producer: query tile, then cache chunks
      // The whole warp walks the items (warp-uniform values, block-table entries read by
      // every lane); one lane arms an item's barrier and one lane per box requests it. The
      // issuing lanes rotate (independent request streams). No L2 prefetch: its requests
      // share this SM's TMA queue with the ring's loads and the P copies, and removing
      // them measured faster (s = 8: 296 -> 270 us; s = 1: 55.0 -> 53.7 us).
      RingPos<S_NR> rp;
      int ic = 0;
      int last[S_NR];
      for (int i = 0; i < S_NR; ++i) last[i] = -1;
      bool ok = true;
      if (ntiles > 0) {
        // first lap: the query tile (chunk-major boxes of CPI chunks, moved into Tensor
        // Memory by the softmax warps, which then free the slots) and q_pe in its own region
        if (lane == 0) {
          mbar_expect_tx(&bars[B_QPE], BM * C::PE_ROW);
          tma_load_2d(sb + C::OFF_QPE, &tm_qpe, 0, qrow0, &bars[B_QPE]);
        }
        for (int qs = 0; qs < C::QS; ++qs) {
          const int slot = rp.slot;
          rp.advance();
          last[slot] = ic++;
          if (lane == 1 + qs) {  // a box's chunks past the last one read as zeros (and count in full)
            mbar_expect_tx(&bars[B_FULL + slot], C::LAT0 * CHUNK);
            tma_load_3d(sb + C::OFF_SRING + slot * C::S_ITEM, &tm_q3, 0, qrow0, qs * C::CPI, &bars[B_FULL + slot]);
          }
          __syncwarp();
        }
      }
      for (int t = 0; ok && t < ntiles; ++t) {
        const int key0 = kstart + t * TK;
        const bool two = kend - key0 > HK;  // the tile's second page holds keys of the chunk
        const int row0 = cache_row(p, bi, key0);
        const int row1 = (PAGED && two) ? cache_row(p, bi, key0 + HK) : 0;
        for (int it = 0; it < C::NITEM; ++it) {
          const int slot = rp.slot;
          const uint32_t prev = rp.phase ^ 1u;
          rp.advance();
          if (ic >= S_NR && !warp_wait(&bars[B_EMPTY + slot], prev, p.wait_ns, abort_flag)) {
            ok = false;
            break;
          }
          const bool has_pe = it == C::NITEM - 1;  // the RoPE chunk is the tile's last
          const uint32_t base = sb + C::OFF_SRING + slot * C::S_ITEM;
          if constexpr (PAGED) {
            const int lb = (ic & 1) * 16;  // first issuing lane of this item
            last[slot] = ic++;
            const uint32_t bytes =
                ((has_pe ? C::LATL * HALF_BOX + C::PE_HALF : C::CPI * HALF_BOX)) * (two ? 2 : 1);
            if (lane == lb) mbar_expect_tx(&bars[B_FULL + slot], bytes);
            __syncwarp();
            const int k = lane - lb;  // box k: chunk it*CPI + k/2 of the tile, page k % 2
            if (k >= 0 && k < 2 * C::CPI && (two || (k & 1) == 0) && it * C::CPI + k / 2 <= C::NBL) {
              const int c = it * C::CPI + k / 2;
              const bool pe = c == C::NBL;
              const uint32_t dst = base + (k / 2) * CHUNK + (k & 1) * (pe ? C::PE_HALF : HALF_BOX);
              const int row = (k & 1) ? row1 : row0;
              if (pe)
                tma_load_2d(dst, &tm_kpe, 0, row, &bars[B_FULL + slot]);
              else
                tma_load_2d(dst, &tm_za, c * 64, row, &bars[B_FULL + slot]);
            }
          } else {
            // one box of the item's latent chunks [128 keys x 64] x LAT (rows past the
            // sequence are read as they are and masked), plus the RoPE box on the last item
            const int lb = (ic & 1) * 2;
            last[slot] = ic++;
            const int lat = has_pe ? C::LATL : C::LAT0;
            if (lane == lb) {
              mbar_expect_tx(&bars[B_FULL + slot], lat * CHUNK + (has_pe ? BM * C::PE_ROW : 0));
              if (lat > 0) tma_load_3d(base, has_pe ? &tm_zb : &tm_za, 0, row0, it * C::CPI, &bars[B_FULL + slot]);
            }
            __syncwarp();
            if (has_pe && lane == lb + 1) tma_load_2d(base + lat * CHUNK, &tm_kpe, 0, row0, &bars[B_FULL + slot]);
          }
          __syncwarp();
        }
      }
      if (lane == 0) {
        if (!ok && !*abort_flag) fail();
        for (int i = 0; i < S_NR; ++i)  // no copy may still be landing when the CTA exits
          if (last[i] >= 0) mbar_wait(&bars[B_FULL + i], (last[i] / S_NR) & 1, kTeardownNs, nullptr);
        if (ntiles > 0) mbar_wait(&bars[B_QPE], 0, kTeardownNs, nullptr);
      }
      __syncwarp();
    } else if (warp == 1) {
      // ------------------------------------------------ MMA issuer: S = Qz Z^T + q_pe K_pe^T
      bool ok = ntiles == 0 || (warp_wait(&bars[B_QREADY], 0, p.wait_ns, abort_flag) &&
                                warp_wait(&bars[B_QPE], 0, p.wait_ns, abort_flag));
      if (ok && ntiles > 0 && p.test_timeout) ok = warp_wait(&bars[B_TEST], 0, kTestWaitNs, abort_flag);
      tc_fence_after();  // Qz was written to Tensor Memory by the softmax warps
      const bool leader = elect_one();
      constexpr uint32_t idS = idesc_bf16_f32(BM, TK, false, false);
      const uint64_t dring = smem_desc(sb + C::OFF_SRING, 16, 1024, kSw128);
      const uint64_t dring_pe = smem_desc(sb + C::OFF_SRING, 16, 8 * C::PE_ROW, C::PE_SWZ);
      const uint64_t dqpe = smem_desc(sb + C::OFF_QPE, 16, 8 * C::PE_ROW, C::PE_SWZ);
      RingPos<S_NR> rp;
      for (int j = 0; j < C::QS; ++j) rp.advance();  // the first lap carried the query tile
      for (int t = 0; ok && t < ntiles; ++t) {
        const int buf = t & 1;
        if (t >= NSB && !warp_wait(&bars[B_SEMPTY + buf], ((t >> 1) - 1) & 1, p.wait_ns, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();  // the softmax warps' loads of this buffer come first
        const uint32_t d_s = tmem + SB0 + buf * TK;
        for (int it = 0; it < C::NITEM; ++it) {
          const int slot = rp.slot;
          const uint32_t ph = rp.phase;
          rp.advance();
          if (!warp_wait(&bars[B_FULL + slot], ph, p.wait_ns, abort_flag)) {
            ok = false;
            break;
          }
          if (leader) {
#pragma unroll
            for (int cc = 0; cc < C::CPI; ++cc) {
              const int j = it * C::CPI + cc;
              const uint64_t so = (uint64_t)((slot * C::S_ITEM + cc * CHUNK) >> 4);
              if (j > C::NBL) {
                // past the RoPE chunk: nothing in this part of the item
              } else if (j < C::NBL) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  tc_mma_ts(d_s, tmem + j * 32 + kk * 8, dring + so + 2 * kk, idS, (j | kk) ? 1u : 0u);
              } else {
#pragma unroll
                for (int kk = 0; kk < P / 16; ++kk) tc_mma_ss(d_s, dqpe + 2 * kk, dring_pe + so + 2 * kk, idS, 1u);
              }
            }
            tc_commit(&bars[B_EMPTY + slot]);
          }
          __syncwarp();
        }
        if (!ok) break;
        if (leader) tc_commit(&bars[B_SFULL + buf]);
        __syncwarp();
      }
      if (lane == 0 && !ok && !*abort_flag) fail();
      if (leader) {  // every issued tcgen05 operation has finished before Tensor Memory is freed
        tc_commit(&bars[B_FIN]);
        mbar_wait(&bars[B_FIN], 0, kTeardownNs, nullptr);
      }
      __syncwarp();
    } else {
      // ------------------------------------------------ query move, softmax, P messages (warps 2-9)
      const int q = warp & 3;            // Tensor Memory lane quadrant this warp may access
      const int hh = (warp - 2) >> 2;    // half of each tile's keys (and of the query boxes) of this warp
      const int r = q * 32 + lane;
      const int row_in_seq = mt * BM + r;
      const bool row_ok = row_in_seq < p.rows;
      const int lim = row_ok ? min(kend, L - p.s + (row_in_seq % p.s) + 1) : 0;  // exclusive key limit
      const uint32_t t_lane = tmem + ((uint32_t)(q * 32) << 16);
      const size_t grow = (size_t)qrow0 + r;
      const bool issuer = warp == 2 && lane == 0;
      float* red = reinterpret_cast<float*>(smem + C::OFF_RED);  // maxima [parity][half][row], then sums [half][row]
      bool ok = ntiles > 0;
      if (ntiles > 0) {
        // Qz row r into Tensor Memory (A operand: lane = row, two bf16 per column, even k
        // low): box j is [128 rows x 64] with 128-byte swizzled rows in ring slot j
        constexpr int JPER = (C::NBL + 1) / 2;
        bool okq = true;
        for (int j = hh * JPER; j < C::NBL && j < (hh + 1) * JPER; ++j) {
          if (!warp_wait(&bars[B_FULL + j / C::CPI], 0, p.wait_ns, abort_flag)) {
            okq = false;
            break;
          }
          const uint8_t* bx = smem + C::OFF_SRING + (j / C::CPI) * C::S_ITEM + (j % C::CPI) * CHUNK + r * 128;
          uint32_t v[32];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint4 x = *reinterpret_cast<const uint4*>(bx + ((u ^ (r & 7)) << 4));
            v[4 * u] = x.x;
            v[4 * u + 1] = x.y;
            v[4 * u + 2] = x.z;
            v[4 * u + 3] = x.w;
          }
          tmem_st32(t_lane + j * 32, v);
        }
        tmem_st_wait();
        tc_fence_before();
        ok = named_bar_and(kBarA, 32 * NSMW, okq && !*abort_flag);
        if (issuer) {
          if (ok) {
            for (int j = 0; j < C::QS; ++j) mbar_arrive(&bars[B_EMPTY + j]);  // the slots may carry cache
            mbar_arrive(&bars[B_QREADY]);
          } else if (!*abort_flag) {
            fail();
          }
        }
      }
      const uint32_t peer_msg0 = mapa_shared(sb + C::OFF_MSG, peer);  // the O CTA's message slots
      const uint32_t peer_pfull0 = mapa_shared(smem_u32(&bars[B_PFULL]), peer);
      float m_ref = -INFINITY, l_run = 0.f;
      for (int t = 0; ok && t < ntiles; ++t) {
        const int buf = t & 1;
        const int m = t & 1;  // message buffer
        const bool okw = warp_wait(&bars[B_SFULL + buf], (t >> 1) & 1, p.wait_ns, abort_flag);
        float x[HK];
        float mx = -INFINITY;
        if (okw) {
          tc_fence_after();
          uint32_t sv[32];
          const uint32_t sbuf = t_lane + SB0 + buf * TK + hh * HK;
          tmem_ld32(sbuf, sv);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) x[c] = __uint_as_float(sv[c]) * p.scale_log2;
          tmem_ld32(sbuf + 32, sv);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) x[32 + c] = __uint_as_float(sv[c]) * p.scale_log2;
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[B_SEMPTY + buf]);  // the buffer may be overwritten
          const int kb = kstart + t * TK + hh * HK;
          if (kb + HK > lim) {
#pragma unroll
            for (int c = 0; c < HK; ++c)
              if (kb + c >= lim) x[c] = -INFINITY;
          }
          float m8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) m8[e] = x[e];
#pragma unroll
          for (int c = 8; c < HK; ++c) m8[c & 7] = fmaxf(m8[c & 7], x[c]);
          mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])), fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
        }
        red[((t & 1) * 2 + hh) * BM + r] = mx;
        if (issuer && t > 0) bulk_wait_read<0>();  // the previous tile's copy has read the staging slot
        // every row warp arrives here on every tile, whatever its wait did, so that all leave
        // the loop together; the other half's maxima are written, and the staging slot is free
        if (!named_bar_and(kBarA, 32 * NSMW, okw && !*abort_flag)) {
          ok = false;
          break;
        }
        mx = fmaxf(mx, red[((t & 1) * 2 + (hh ^ 1)) * BM + r]);
        float alpha = 1.f;
        if (mx > m_ref + kRescaleLog2) {  // both halves of a row take the same decision
          alpha = fast_exp2(m_ref - mx);  // 0 when nothing was seen yet
          m_ref = mx;
          l_run *= alpha;
        }
        const float mneg = m_ref == -INFINITY ? 0.f : -m_ref;  // all keys masked so far: x = -inf -> 0
        uint32_t pk[HK / 2];
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int e = 0; e < HK / 2; ++e) {
          const float p0 = fast_exp2(x[2 * e] + mneg);
          const float p1 = fast_exp2(x[2 * e + 1] + mneg);
          ps[e & 3] += p0 + p1;
          pk[e] = pack_bf16(p0, p1);
        }
        l_run += (ps[0] + ps[1]) + (ps[2] + ps[3]);
        // P row r, keys of this half, into staging slot m: K-block hh of [128 rows x 64 keys],
        // 128-byte rows, 16-byte unit u at (u ^ (r & 7))
        uint8_t* st = smem + C::OFF_STG;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          *reinterpret_cast<uint4*>(st + hh * P_BLK + r * 128 + ((u ^ (r & 7)) << 4)) =
              make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        if (hh == 0) {
          // the first tile fills an empty O (its MMAs do not accumulate): nothing to rescale
          const float a_out = t == 0 ? 1.f : alpha;
          reinterpret_cast<float*>(st + MSG_ALPHA)[r] = a_out;
          const bool any = __any_sync(0xffffffffu, a_out != 1.f);
          if (lane == 0) reinterpret_cast<int*>(st + MSG_FLAGS)[q] = any ? 1 : 0;
        }
        fence_proxy_async_smem();  // the bulk copy (async proxy) reads what these stores wrote
        named_bar_sync(kBarB, 32 * NSMW);
        if (issuer) {
          // the O CTA's MMAs are done with its message buffer m (tile t - NMSG)
          const bool free_ok =
              t < NMSG || mbar_wait(&bars[B_PFREE + m], ((t >> 1) - 1) & 1, p.wait_ns, abort_flag);
          if (free_ok) {
            // in pieces of ~2 KB: the SM's TMA engine then serves the ring's loads between
            // them instead of behind the whole 33 KB (measured, same box: 16 pieces 50.5 vs
            // 52.8 us at s = 1 and 77.4 vs 82.0 at s = 2, s = 8 within 1 %; 32 or 64 pieces
            // are slower, the issue cost per piece dominating)
            for (uint32_t o = 0; o < (uint32_t)MSG_BYTES; o += kMsgPiece) {
              const uint32_t nb = (uint32_t)MSG_BYTES - o < kMsgPiece ? (uint32_t)MSG_BYTES - o : kMsgPiece;
              bulk_copy_to_peer(peer_msg0 + m * MSG_STRIDE + o, sb + C::OFF_STG + o, nb, peer_pfull0 + m * 8);
            }
            bulk_commit();
          } else if (!*abort_flag) {
            fail();
          }
        }
      }
      ok = named_bar_and(kBarA, 32 * NSMW, ok && !*abort_flag);
      red[(4 + hh) * BM + r] = l_run;
      named_bar_sync(kBarB, 32 * NSMW);
      const float l_tot = red[4 * BM + r] + red[5 * BM + r];
      if (ok && hh == 0) {
        if (row_ok) {
          const float lse = l_tot > 0.f ? (m_ref + log2f(l_tot)) * kLn2 : -INFINITY;
          if (whole) {
            if (p.lse) p.lse[grow] = lse;
          } else {
            p.ws_lse[(part_row0 + r) * part_n + split] = lse;
          }
        }
        reinterpret_cast<float*>(smem + C::OFF_FIN)[r] = l_tot > 0.f ? 1.f / l_tot : 0.f;
        fence_proxy_async_smem();
      }
      named_bar_sync(kBarA, 32 * NSMW);
      if (issuer) {
        if (ok) {
          bulk_copy_to_peer(mapa_shared(sb + C::OFF_FIN, peer), sb + C::OFF_FIN, FIN_BYTES,
                            mapa_shared(smem_u32(&bars[B_FINFULL]), peer));
          bulk_commit();
        }
        bulk_wait<0>();  // every copy into the peer has landed
        // the O CTA's last commits into this CTA's barriers have arrived
        if (ok)
          for (int t = ntiles > NMSG ? ntiles - NMSG : 0; t < ntiles; ++t)
            if (!mbar_wait(&bars[B_PFREE + (t & 1)], (t >> 1) & 1, p.wait_ns, abort_flag)) {
              if (!*abort_flag) fail();
              break;
            }
      }
    }
  } else {
    // =====================================================================================
    // O CTA
    if (warp == 0) {
      // ------------------------------------------------ producer: Z slabs into the O-ring
      RingPos<O_NR> rp;
      int ic = 0;
      int last[O_NR];
      for (int i = 0; i < O_NR; ++i) last[i] = -1;
      bool ok = true;
      for (int t = 0; ok && t < ntiles; ++t) {
        const int key0 = kstart + t * TK;
        const int nkh = kend - key0 > HK ? 2 : 1;
        for (int kh = 0; ok && kh < nkh; ++kh) {
          const int row0 = cache_row(p, bi, key0 + kh * HK);
          for (int nh = 0; nh < C::NH; ++nh) {
            const int slot = rp.slot;
            const uint32_t prev = rp.phase ^ 1u;
            rp.advance();
            if (ic >= O_NR && !warp_wait(&bars[B_EMPTY + slot], prev, p.wait_ns, abort_flag)) {
              ok = false;
              break;
            }
            last[slot] = ic;
            if (lane == (ic & 1)) {  // one box per item; the issuing lane alternates
              mbar_expect_tx(&bars[B_FULL + slot], C::O_ITEM);
              tma_load_3d(sb + C::OFF_ORING + slot * C::O_ITEM, &tm_zo, 0, row0, nh * (C::ON / 64), &bars[B_FULL + slot]);
            }
            ++ic;
            __syncwarp();
          }
        }
      }
      if (lane == 0) {
        if (!ok && !*abort_flag) fail();
        for (int i = 0; i < O_NR; ++i)
          if (last[i] >= 0) mbar_wait(&bars[B_FULL + i], (last[i] / O_NR) & 1, kTeardownNs, nullptr);
      }
      __syncwarp();
    } else if (warp == 1) {
      // ------------------------------------------------ MMA issuer: O += P Z
      const bool leader = elect_one();
      constexpr uint32_t idO = idesc_bf16_f32(BM, C::ON, false, true);
      const uint64_t dmsg = smem_desc(sb + C::OFF_MSG, 16, 1024, kSw128);       // P, K-major
      const uint64_t dz = smem_desc(sb + C::OFF_ORING, HALF_BOX, 1024, kSw128);  // Z slab, MN-major
      RingPos<O_NR> rp;
      int ncorr = 0;
      bool ok = true;
      for (int t = 0; ok && t < ntiles; ++t) {
        const int m = t & 1;
        if (leader) mbar_expect_tx(&bars[B_PFULL + m], MSG_BYTES);  // this use's one arrival + bytes
        __syncwarp();
        if (!warp_wait(&bars[B_PFULL + m], (t >> 1) & 1, p.wait_ns, abort_flag)) {
          ok = false;
          break;
        }
        const volatile int* fl = reinterpret_cast<const volatile int*>(msg(m) + MSG_FLAGS);
        const bool rescale = t > 0 && (fl[0] | fl[1] | fl[2] | fl[3]) != 0;
        if (rescale) {
          // every O MMA issued so far (tiles < t) must be complete first: a commit made now
          // tracks exactly those (one commit and one wait per rescale, so the waits follow
          // the barrier's phases one by one)
          if (leader) tc_commit(&bars[B_ODONE]);
          __syncwarp();
          if (!warp_wait(&bars[B_ODONE], ncorr & 1, p.wait_ns, abort_flag)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            *req_tile = t;
            mbar_arrive(&bars[B_CREQ]);
          }
          __syncwarp();
          if (!warp_wait(&bars[B_CDONE], ncorr & 1, p.wait_ns, abort_flag)) {
            ok = false;
            break;
          }
          ++ncorr;
          tc_fence_after();  // the rescaled O (tcgen05.st of the row warps) comes first
        }
        const int key0 = kstart + t * TK;
        const int nkh = kend - key0 > HK ? 2 : 1;
        for (int kh = 0; ok && kh < nkh; ++kh) {
          for (int nh = 0; nh < C::NH; ++nh) {
            const int slot = rp.slot;
            const uint32_t ph = rp.phase;
            rp.advance();
            if (!warp_wait(&bars[B_FULL + slot], ph, p.wait_ns, abort_flag)) {
              ok = false;
              break;
            }
            const int first_bad = L - (key0 + kh * HK);  // rows at or past the sequence end may hold anything
            if (first_bad < HK) {
              uint8_t* item = smem + C::OFF_ORING + slot * C::O_ITEM;
              const int nrow = HK - first_bad;
              for (int idx = lane; idx < nrow * (C::ON / 64) * 8; idx += 32) {
                const int rr = first_bad + idx / ((C::ON / 64) * 8);
                const int rem = idx % ((C::ON / 64) * 8);
                *reinterpret_cast<uint4*>(item + (rem / 8) * HALF_BOX + rr * 128 + (rem % 8) * 16) =
                    make_uint4(0, 0, 0, 0);
              }
              fence_proxy_async_smem();
              __syncwarp();
            }
            if (leader) {
              const uint64_t a0 = dmsg + (uint64_t)((m * MSG_STRIDE + kh * P_BLK) >> 4);
              const uint64_t b0 = dz + (uint64_t)((slot * C::O_ITEM) >> 4);
#pragma unroll
              for (int kk = 0; kk < HK / 16; ++kk)
                tc_mma_ss(tmem + nh * C::ON, a0 + 2 * kk, b0 + (uint64_t)((kk * 16 * 128) >> 4), idO,
                          (t > 0 || kh > 0 || kk > 0) ? 1u : 0u);
              tc_commit(&bars[B_EMPTY + slot]);
            }
            __syncwarp();
          }
        }
        if (!ok) break;
        if (leader) tc_commit_multicast(&bars[B_PFREE + m], (uint16_t)(1u << kRankS));  // S may refill buffer m
        __syncwarp();
      }
      if (leader && ok && ntiles > 0) tc_commit(&bars[B_OFINAL]);
      if (lane == 0) {
        if (!ok && !*abort_flag) fail();
        *req_tile = -1;  // end marker for the row warps
        mbar_arrive(&bars[B_CREQ]);
      }
      if (leader) {
        tc_commit(&bars[B_FIN]);
        mbar_wait(&bars[B_FIN], 0, kTeardownNs, nullptr);
      }
      __syncwarp();
    } else {
      // ------------------------------------------------ rescale requests, then the epilogue
      const int q = warp & 3;
      const int hh = (warp - 2) >> 2;  // half of the output columns of this warp
      const int r = q * 32 + lane;
      const int c_lo = hh * C::OCOLS;
      const uint32_t t_lane = tmem + ((uint32_t)(q * 32) << 16);
      bool ok = true;
      for (int k = 0;; ++k) {
        if (!warp_wait(&bars[B_CREQ], k & 1, p.wait_ns, abort_flag)) {
          ok = false;
          break;
        }
        const int tile = *req_tile;
        if (tile < 0) break;
        const float alpha = reinterpret_cast<const volatile float*>(msg(tile & 1) + MSG_ALPHA)[r];
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
          tc_fence_after();
#pragma unroll 1
          for (int c0 = c_lo; c0 < c_lo + C::OCOLS; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(t_lane + c0, v);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 32; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * alpha);
            tmem_st32(t_lane + c0, v);
          }
          tmem_st_wait();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[B_CDONE]);
      }
      if (ok && ntiles > 0 && !*abort_flag) {
        ok = warp_wait(&bars[B_OFINAL], 0, p.wait_ns, abort_flag) &&
             warp_wait(&bars[B_FINFULL], 0, p.wait_ns, abort_flag);
        if (!ok) {
          if (lane == 0 && !*abort_flag) fail();
        } else {
          tc_fence_after();
          const float inv = reinterpret_cast<const float*>(smem + C::OFF_FIN)[r];
          // O / l of this warp's 32 rows x OCOLS columns: Tensor Memory -> registers (up to
          // four 32-column loads in flight per wait) -> bf16 rows staged in shared memory (the
          // O-ring, idle once every MMA has completed; 16-byte units XOR-swizzled by the row,
          // so that neither the row-per-lane writes nor the unit-per-lane reads conflict) ->
          // whole row segments stored to global memory, 16 bytes per lane.
          constexpr int UNITS = C::OCOLS / 8;  // 16-byte bf16 units per row of this warp
          constexpr int ROWB = C::OCOLS * 2;
          constexpr int RPI = 32 / UNITS;      // rows per store instruction
          constexpr int GRP = C::OCOLS / 32 < 4 ? C::OCOLS / 32 : 4;  // 32-column loads per wait
          uint8_t* stg = smem + C::OFF_ORING + (warp - 2) * 32 * ROWB;
#pragma unroll 1
          for (int g0 = 0; g0 < C::OCOLS; g0 += 32 * GRP) {
            uint32_t v[GRP][32];
#pragma unroll
            for (int gi = 0; gi < GRP; ++gi) tmem_ld32(t_lane + c_lo + g0 + gi * 32, v[gi]);
            tmem_ld_wait();
#pragma unroll
            for (int gi = 0; gi < GRP; ++gi) {
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int u = (g0 + gi * 32) / 8 + e;
                const uint32_t* w = v[gi] + 8 * e;
                *reinterpret_cast<uint4*>(stg + lane * ROWB + ((u ^ (lane % UNITS)) << 4)) =
                    make_uint4(pack_bf16(__uint_as_float(w[0]) * inv, __uint_as_float(w[1]) * inv),
                               pack_bf16(__uint_as_float(w[2]) * inv, __uint_as_float(w[3]) * inv),
                               pack_bf16(__uint_as_float(w[4]) * inv, __uint_as_float(w[5]) * inv),
                               pack_bf16(__uint_as_float(w[6]) * inv, __uint_as_float(w[7]) * inv));
              }
            }
          }
          __syncwarp();
          const int ju = lane % UNITS;
#pragma unroll 4
          for (int rr = lane / UNITS; rr < 32; rr += RPI) {
            const int rs = q * 32 + rr;  // row within the tile
            if (mt * BM + rs >= p.rows) continue;
            const uint4 xv = *reinterpret_cast<const uint4*>(stg + rr * ROWB + ((ju ^ (rr % UNITS)) << 4));
            const size_t g = (size_t)qrow0 + rs;
            __nv_bfloat16* dst = whole ? p.o_lat + g * KL : p.ws_ob + ((part_row0 + rs) * part_n + split) * KL;
            *reinterpret_cast<uint4*>(dst + c_lo + ju * 8) = xv;
          }
        }
      }
    }
  }

  // ---- teardown: nothing of this CTA is in flight; the peer leaves at the same time
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// host side: tensor maps and launch

CUtensorMapSwizzle swizzle_for(int row_bytes) {
  return row_bytes >= 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                          : (row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
}

// 2-D bf16 map over a [rows, cols] row-major matrix with boxes [box_rows, box_cols]
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows, uint32_t box_cols) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  return encode_tmap_bf16(m, base, 2, dims, strides, box, swizzle_for((int)box_cols * 2));
}

// 3-D view {64 columns, rows, cols/64 chunks} of a [rows, cols] bf16 matrix (row stride cols*2
// bytes, chunk stride 128 bytes) with boxes {64, box_rows, box_chunks}: a box lands chunk-major,
// [box_chunks][box_rows][64], each 128-byte row swizzled
bool make_chunk_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                    uint32_t box_chunks) {
  const cuuint64_t dims[3] = {64, rows, cols / 64};
  const cuuint64_t strides[2] = {cols * 2, 128};
  const cuuint32_t box[3] = {64, box_rows, box_chunks};
  return encode_tmap_bf16(m, base, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int KL, int P, bool PAGED>
cudaError_t launch_klp(const MlaLaunch& a, cudaStream_t stream) {
  using C = MlaCfg<KL, P>;
  static std::atomic<unsigned long long> smem_limit_set{0};
  if (cudaError_t e = ensure_smem_limit(mla_pair_kernel<KL, P, PAGED>, C::SMEM, smem_limit_set)) return e;
  const uint64_t krows = a.paged ? (uint64_t)a.num_pages * 64 : (uint64_t)a.b * a.capacity;
  const uint64_t qrows = (uint64_t)a.b * a.h * a.s;
  CUtensorMap tq3, tqpe, tza, tzb, tkpe, tzo;
  bool ok = make_chunk_map(&tq3, a.qz, qrows, KL, BM, C::LAT0) && make_map(&tqpe, a.q_pe, qrows, P, BM, P) &&
            make_chunk_map(&tzo, a.z, krows, KL, HK, C::ON / 64);
  if (PAGED) {
    ok = ok && make_map(&tza, a.z, krows, KL, HK, 64) && make_map(&tkpe, a.k_pe, krows, P, HK, P);
    tzb = tza;
  } else {
    ok = ok && make_chunk_map(&tza, a.z, krows, KL, TK, C::LAT0) && make_chunk_map(&tzb, a.z, krows, KL, TK, C::LATL > 0 ? C::LATL : 1) &&
         make_map(&tkpe, a.k_pe, krows, P, TK, P);
  }
  if (!ok) return cudaErrorInvalidValue;
  MlaParams p;
  p.ws_ob = static_cast<__nv_bfloat16*>(a.ws_o);
  p.seqlens = a.seqlens;
  p.block_table = a.block_table;
  p.max_pages = a.max_pages;
  p.paged = a.paged;
  p.capacity = a.capacity;
  p.num_pages = a.num_pages;
  p.b = a.b;
  p.s = a.s;
  p.h = a.h;
  p.rows = a.h * a.s;
  p.nsplit = a.nsplit;
  p.chunk = a.chunk;
  p.scale_log2 = a.scale * kLog2e;
  p.o_lat = static_cast<__nv_bfloat16*>(a.o_lat);
  p.lse = a.lse;
  p.ws_lse = a.ws_lse;
  p.err = a.err;
  p.wait_ns = a.wait_ns;
  p.test_timeout = a.test_timeout;
  const int mtiles = (p.rows + BM - 1) / BM;
  p.mtiles = mtiles;
  p.tail_whole = a.tail_whole;
  p.tail_k = a.tail_k;
  p.tail_chunk = a.tail_chunk;
  // a cluster of two CTAs per row tile, launched as a programmatic dependent
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = a.tail_k > 0 ? dim3(2 * (a.tail_whole + a.tail_units * a.tail_k)) : dim3(2 * mtiles, a.nsplit, a.b);
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, mla_pair_kernel<KL, P, PAGED>, tq3, tqpe, tza, tzb, tkpe, tzo, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int KL, int P>
cudaError_t launch_kl(const MlaLaunch& a, cudaStream_t stream) {
  return a.paged ? launch_klp<KL, P, true>(a, stream) : launch_klp<KL, P, false>(a, stream);
}

}  // namespace

int mla_ctas_per_row_tile() { return 2; }
int mla_tile_keys() { return TK; }
bool mla_supported(int k, int p) { return (k == 512 && p == 64) || (k == 64 && p == 16); }

cudaError_t launch_mla_latent(const MlaLaunch& a, cudaStream_t stream) {
  if (a.k == 512 && a.p == 64) return launch_kl<512, 64>(a, stream);
  if (a.k == 64 && a.p == 16) return launch_kl<64, 16>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace decattn
