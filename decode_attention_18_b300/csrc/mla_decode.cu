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
// Kernel design (one CTA = 128 query rows x one context chunk x one half of the
// output columns):
//   * All h*s query rows of a sequence are packed into the MMA M dimension
//     (row = head*s + token), 128 rows per CTA.
//   * Q' = [Qz | q_pe] stays in shared memory for the whole chunk. The cache
//     is consumed in tiles of 128 latent rows. One ring of 16 KB slots carries,
//     in exactly the order the MMAs consume them, the tile's 64-wide column
//     chunks [128 rows x 64] (plus the RoPE chunk), each loaded by TMA as two
//     64-row boxes (a box never crosses a 64-token page), and the O slab
//     pairs: the CTA's own output columns of 32 latent rows, re-read from L2.
//   * tcgen05.mma (kind::f16, bf16 in, fp32 accumulate in Tensor Memory):
//       S  = Q' K'^T    M=128, N=128 keys, K=k+p   (both operands in smem)
//       O += P Z_half   M=128, N=256 cols, K=16 keys per slab, with P read
//                       from Tensor Memory and the Z slab (MN-major) from smem
//     The fp32 accumulator of 128 rows x k = 512 columns would fill all of
//     TMEM, so the output columns are split over 2 CTAs per row tile, each
//     recomputing S for the same rows. TMEM holds O (256 columns) and two
//     128-column S buffers; the softmax writes P (bf16, two per column) over
//     the first 64 columns of its own S buffer, so P is double-buffered too.
//   * The O MMAs of tile t are issued interleaved with the S MMAs of tile
//     t+1, so the tensor pipe stays busy while the softmax of tile t runs.
//     tcgen05 MMAs of one thread execute in issue order, so the S of tile t+2
//     (same buffer) never overtakes the O MMAs still reading P of tile t.
//   * Softmax: two warps per TMEM lane quadrant (thread = row, 64 keys each);
//     they exchange row maxima through shared memory and keep one reference
//     maximum per row that moves only when the row maximum grows by more than
//     2^8 (O is then rescaled in TMEM). Exponentials use ex2.approx.
//   * Warp roles: warp 0 issues the TMA loads, warp 1 the MMAs (the warp
//     zeroes tails and owns the TMEM allocation), warps 2-9 run the softmax
//     and the epilogue. The producer and the MMA issuer handle every ring item
//     one after another, so their per-item cost sets the pace: each whole warp
//     computes the item's operands (warp-uniform values), one elected lane
//     issues, an already completed barrier costs one test, and the TMEM base
//     is a constant (the CTA owns all 512 columns).
//   * Latent rows past the sequence end may hold anything: slabs wholly past
//     it are not multiplied; a slab that straddles it has its rows past the
//     end zeroed before the O MMA, so P Z stays finite.
//   * Every mbarrier wait is bounded; on time-out the CTA records the error,
//     stops issuing work, waits for its own copies and MMAs, frees TMEM and
//     returns.
//   * Launched as a programmatic dependent of the previous kernel on the
//     stream: barrier set-up, TMEM allocation and tensor-map prefetch run
//     before griddepcontrol.wait, every global read after it.
// Output: with a single chunk, bf16 O_lat and the LSE directly; otherwise fp32
// partials (O / l, LSE) merged by the combine kernel. Either way O / l is
// staged in shared memory (free once the last MMA has completed) and stored as
// whole row segments.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"

namespace decattn {

namespace {

constexpr int TK = 128;         // latent rows (keys) per S tile
constexpr int NR = 5;           // ring slots (16 KB each)
constexpr int SLAB = 16;        // keys per O slab (= MMA K)
constexpr int PAIR = 2 * SLAB;  // keys per O ring item
constexpr int BMROWS = 128;     // query rows per CTA (MMA M)
constexpr int NSMW = 8;         // softmax warps
constexpr int NTHREADS = 32 * (2 + NSMW);
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.f;                        // move the reference max only past 2^8
constexpr unsigned long long kTeardownNs = 1000000000ull;  // 1 s for own copies / MMAs at exit
constexpr unsigned long long kTestWaitNs = 1000000ull;     // 1 ms forced-timeout wait

constexpr int align1024(int x) { return (x + 1023) & ~1023; }
constexpr int pow2_cols(int x) { return x <= 32 ? 32 : (x <= 64 ? 64 : (x <= 128 ? 128 : (x <= 256 ? 256 : 512))); }

struct MlaParams {
  const int32_t* seqlens;
  const int32_t* block_table;
  int max_pages, paged, capacity, num_pages;
  int b, s, h, rows, nsplit, chunk;
  float scale_log2;
  __nv_bfloat16* o_lat;
  float* lse;
  float* ws_o;
  float* ws_lse;
  unsigned* err;
  unsigned long long wait_ns;
  int test_timeout;
};

template <int KL, int P>
struct MlaCfg {
  static constexpr int NH = KL >= 512 ? 2 : 1;  // CTAs per 128-row tile (output-column halves)
  static constexpr int KLH = KL / NH;           // O columns per CTA
  static constexpr int NBL = KL / 64;           // 64-wide latent column chunks
  static constexpr int NCH = NBL + 1;           // + the RoPE chunk
  static constexpr int J0 = NCH > 5 ? 5 : NCH - 1;  // O items of the previous tile start after chunk J0
  static constexpr int PE_ROW = P * 2;          // bytes per RoPE row
  static constexpr uint32_t PE_SWZ = PE_ROW == 128 ? kSw128 : (PE_ROW == 64 ? kSw64 : kSw32);
  static constexpr int Q_BOX = BMROWS * 128;
  static constexpr int Q_LAT = NBL * Q_BOX;
  static constexpr int Q_PE = BMROWS * PE_ROW;
  static constexpr int SLOT = TK * 128;               // ring slot: one [128 keys x 64] chunk
  static constexpr int HALF_LAT = 64 * 128;           // one 64-row box of a latent chunk
  static constexpr int HALF_PE = 64 * PE_ROW;         // one 64-row box of the RoPE chunk
  static constexpr int PBOX = PAIR * 128;             // [32 keys x 64 cols] box of an O item
  static constexpr int PAIR_BYTES = (KLH / 64) * PBOX;
  static constexpr int OFF_QPE = Q_LAT;
  static constexpr int OFF_RING = align1024(Q_LAT + Q_PE);
  static constexpr int OFF_RED = OFF_RING + NR * SLOT;          // row-max exchange [2][2][128] floats
  static constexpr int OFF_BAR = align1024(OFF_RED + 2 * 2 * BMROWS * 4);
  // + barriers. No alignment slack: the dynamic window follows the CTA's 1 KB reserved
  // shared memory and is 1024-byte aligned; the kernel checks this and refuses otherwise.
  static constexpr int SMEM = OFF_BAR + 512;
  static constexpr int TM_S = KLH;                   // two S buffers after the O accumulator
  static constexpr int TM_COLS = pow2_cols(KLH + 2 * TK);
  static_assert(KL % 64 == 0 && KLH % 64 == 0 && KLH <= 256, "latent width");
  static_assert(P % 16 == 0 && PE_ROW <= 128, "rope width");
  static_assert(PAIR_BYTES <= SLOT, "O item fits a ring slot");
  static_assert(SMEM <= 232448, "shared memory");
  static_assert(KLH + 2 * TK <= 512, "tensor memory");
};

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
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, limit_ns, abort_flag));
}

// same, with a cheap first test for the common case of a phase that already completed
__device__ __forceinline__ bool warp_wait_fast(uint64_t* bar, uint32_t parity, uint64_t limit_ns,
                                               volatile int* abort_flag) {
  if (__all_sync(0xffffffffu, mbar_test(bar, parity))) return true;
  return warp_wait(bar, parity, limit_ns, abort_flag);
}

// position in the ring: next slot and the phase parity of its current use
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

// The ring's item sequence, shared by the producer and the MMA issuer:
// iteration u (0..ntiles) carries the NCH chunks of tile u (u < ntiles) with
// the O items (32-key slab pairs) of tile u-1 spread over chunks J0..NCH-1;
// the last iteration carries only the O items of the last tile.
template <int NCH, int J0, class Chunk, class Pair>
__device__ __forceinline__ bool walk_iteration(int u, int ntiles, int npairs_prev, Chunk&& chunk, Pair&& pair) {
  if (u >= ntiles) {
    for (int q = 0; q < npairs_prev; ++q)
      if (!pair(u - 1, q)) return false;
    return true;
  }
  int done = 0;
  for (int j = 0; j < NCH; ++j) {
    if (!chunk(u, j)) return false;
    if (npairs_prev > 0 && j >= J0) {
      const int target = (npairs_prev * (j - J0 + 1) + (NCH - J0) - 1) / (NCH - J0);
      for (; done < target; ++done)
        if (!pair(u - 1, done)) return false;
    }
  }
  return true;
}

template <int KL, int P>
__global__ void __launch_bounds__(NTHREADS, 1)
    mla_latent_kernel(const __grid_constant__ CUtensorMap tm_qz, const __grid_constant__ CUtensorMap tm_qpe,
                      const __grid_constant__ CUtensorMap tm_z64, const __grid_constant__ CUtensorMap tm_kpe64,
                      const __grid_constant__ CUtensorMap tm_z32, MlaParams p) {
  using C = MlaCfg<KL, P>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sb = smem_u32(smem);
  if (sb & 1023u) {  // 128-byte swizzled tiles need 1024-byte aligned slots
    if (threadIdx.x == 0) raise_error(p.err, kErrLaunch);
    return;
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int lh = blockIdx.x % C::NH;
  const int mt = blockIdx.x / C::NH;
  const int split = blockIdx.y;
  const int bi = blockIdx.z;
  const int kstart = split * p.chunk;
  const int qrow0 = bi * p.rows + mt * BMROWS;  // first flattened [b*h*s] query row

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_box = bars + 32;     // [NCH] box j of the query tile Q' landed
  uint64_t* r_full = bars + 1;     // [NR] ring item landed
  uint64_t* r_empty = bars + 6;    // [NR] ring item consumed by its MMAs
  uint64_t* s_ready = bars + 11;   // [2]  S tile in TMEM (and the previous tile's O MMAs complete)
  uint64_t* p_full = bars + 13;    //      P in TMEM (+ O rescaled)
  uint64_t* o_final = bars + 14;   //      last O MMAs complete
  uint64_t* test_bar = bars + 15;
  uint64_t* fin_bar = bars + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 17);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 18);
  float* red = reinterpret_cast<float*>(smem + C::OFF_RED);  // [parity][column half][row]
  volatile int* okf = reinterpret_cast<volatile int*>(bars + 20);  // [parity][column half][quadrant]

  // Set-up that touches no global memory (it overlaps the end of the previous kernel
  // when the launch allows it).
  if (threadIdx.x == 0) {
    for (int j = 0; j < C::NCH; ++j) mbar_init(&q_box[j], 1);
    for (int i = 0; i < NR; ++i) {
      mbar_init(&r_full[i], 1);
      mbar_init(&r_empty[i], 1);
    }
    mbar_init(&s_ready[0], 1);
    mbar_init(&s_ready[1], 1);
    mbar_init(p_full, NSMW);  // one arrival per softmax warp
    mbar_init(o_final, 1);
    mbar_init(test_bar, 1);  // never signalled: the forced-timeout test waits on it
    mbar_init(fin_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_qz);
    prefetch_tmap(&tm_qpe);
    prefetch_tmap(&tm_z64);
    prefetch_tmap(&tm_kpe64);
    prefetch_tmap(&tm_z32);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // The CTA allocates all 512 columns, so its allocation can only start at lane 0,
  // column 0. The kernel uses that address as a constant (operands known to be
  // warp-uniform keep tcgen05 issue cheap) and checks it here.
  static_assert(C::TM_COLS == 512, "whole-TMEM allocation");
  constexpr uint32_t tmem = 0;
  const bool tmem_ok = *tmem_slot == tmem;
  if (!tmem_ok && threadIdx.x == 0) raise_error(p.err, kErrLaunch);

  // inputs written by earlier kernels (queries, cache, lengths) are read from here on
  pdl_wait();
  pdl_trigger();
  const int L = p.seqlens[bi];
  const bool active = kstart < L;  // a chunk past the end does nothing (the combine skips it)
  if (!active && L <= 0 && p.nsplit == 1) {  // empty sequence without a combine pass: zero rows, LSE = -inf
    for (int idx = threadIdx.x; idx < BMROWS * (C::KLH / 8); idx += blockDim.x) {
      const int r = idx / (C::KLH / 8);
      if (mt * BMROWS + r >= p.rows) continue;
      const size_t grow = (size_t)bi * p.rows + mt * BMROWS + r;
      *reinterpret_cast<uint4*>(p.o_lat + grow * KL + lh * C::KLH + (idx % (C::KLH / 8)) * 8) =
          make_uint4(0, 0, 0, 0);
      if (p.lse && lh == 0 && idx % (C::KLH / 8) == 0) p.lse[grow] = -INFINITY;
    }
  }
  const int kend = min(L, kstart + p.chunk);
  const int ntiles = active ? (kend - kstart + TK - 1) / TK : 0;
  auto tile_keys = [&](int t) { return min(TK, kend - (kstart + t * TK)); };
  auto tile_slabs = [&](int t) { return (tile_keys(t) + SLAB - 1) / SLAB; };
  auto tile_pairs = [&](int t) { return t >= 0 ? (tile_keys(t) + PAIR - 1) / PAIR : 0; };

  auto fail = [&]() {
    raise_error(p.err, kErrWaitTimeout);
    *abort_flag = 1;
  };

  if (!tmem_ok || !active) {
    // nothing to issue; fall through to the deallocation
  } else if (warp == 0) {
    // ------------------------------------------------------------ producer: TMA into the ring
    // The whole warp walks the item sequence and computes every coordinate (warp-uniform
    // values, block-table entries read by all lanes); one elected lane issues the copies.
    const uint64_t pol_last = policy_evict_first();  // O items are the last reads of those rows
    const bool leader = elect_one();
    int last[NR];
    for (int i = 0; i < NR; ++i) last[i] = -1;
    // Q' box j is requested just before the first tile's chunk j (each on its own barrier),
    // so the first S MMAs start as soon as their two boxes have landed instead of after the
    // whole 144 KB query tile.
    int qb_issued = 0;
    int ic = 0;  // ring items issued
    RingPos rp;
    auto acquire = [&](int& slot) -> bool {
      slot = rp.slot;
      const uint32_t prev = rp.phase ^ 1u;  // phase of the slot's previous use
      rp.advance();
      if (ic >= NR && !warp_wait_fast(&r_empty[slot], prev, p.wait_ns, abort_flag)) return false;
      last[slot] = ic;
      ++ic;
      return true;
    };
    auto chunk = [&](int u, int j) -> bool {
      if (u == 0) {
        if (leader) {
          if (j == C::NBL) {
            mbar_expect_tx(&q_box[j], C::Q_PE);
            tma_load_2d(sb + C::OFF_QPE, &tm_qpe, 0, qrow0, &q_box[j]);
          } else {
            mbar_expect_tx(&q_box[j], C::Q_BOX);
            tma_load_2d(sb + j * C::Q_BOX, &tm_qz, j * 64, qrow0, &q_box[j]);
          }
        }
        __syncwarp();
        qb_issued = j + 1;
      }
      int slot;
      if (!acquire(slot)) return false;
      const int key0 = kstart + u * TK;
      const bool two = tile_keys(u) > 64;
      const int row0 = cache_row(p, bi, key0);
      const int row1 = two ? cache_row(p, bi, key0 + 64) : 0;
      const uint32_t dst = sb + C::OFF_RING + slot * C::SLOT;
      if (leader) {
        if (j == C::NBL) {
          mbar_expect_tx(&r_full[slot], C::HALF_PE * (two ? 2 : 1));
          tma_load_2d(dst, &tm_kpe64, 0, row0, &r_full[slot]);
          if (two) tma_load_2d(dst + C::HALF_PE, &tm_kpe64, 0, row1, &r_full[slot]);
        } else {
          mbar_expect_tx(&r_full[slot], C::HALF_LAT * (two ? 2 : 1));
          tma_load_2d(dst, &tm_z64, j * 64, row0, &r_full[slot]);
          if (two) tma_load_2d(dst + C::HALF_LAT, &tm_z64, j * 64, row1, &r_full[slot]);
        }
      }
      __syncwarp();
      return true;
    };
    auto pair = [&](int v, int q) -> bool {
      int slot;
      if (!acquire(slot)) return false;
      const uint32_t dst = sb + C::OFF_RING + slot * C::SLOT;
      const int row = cache_row(p, bi, kstart + v * TK + q * PAIR);
      if (leader) {
        mbar_expect_tx(&r_full[slot], C::PAIR_BYTES);
#pragma unroll
        for (int k = 0; k < C::KLH / 64; ++k)
          tma_load_2d_hint(dst + k * C::PBOX, &tm_z32, lh * C::KLH + k * 64, row, &r_full[slot], pol_last);
      }
      __syncwarp();
      return true;
    };
    bool ok = true;
    for (int u = 0; ok && u <= ntiles; ++u)
      ok = walk_iteration<C::NCH, C::J0>(u, ntiles, tile_pairs(u - 1), chunk, pair);
    if (lane == 0) {
      if (!ok && !*abort_flag) fail();
      // no copy may still be landing in shared memory when the CTA exits
      for (int j = 0; j < qb_issued; ++j) mbar_wait(&q_box[j], 0, kTeardownNs, nullptr);
      for (int i = 0; i < NR; ++i)
        if (last[i] >= 0) mbar_wait(&r_full[i], (last[i] / NR) & 1, kTeardownNs, nullptr);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (one elected lane issues; the warp zeroes tails)
    bool ok = true;
    if (p.test_timeout) ok = warp_wait(test_bar, 0, kTestWaitNs, abort_flag);
    const bool leader = elect_one();
    constexpr uint32_t idS = idesc_bf16_f32(BMROWS, TK, false, false);
    constexpr uint32_t idO = idesc_bf16_f32(BMROWS, C::KLH, false, true);
    // descriptors of the resident Q' chunks and of ring slot 0 (start-address field advanced per slot / k step)
    const uint64_t dq0 = smem_desc(sb, 16, 1024, kSw128);
    const uint64_t dqpe = smem_desc(sb + C::OFF_QPE, 16, 8 * C::PE_ROW, C::PE_SWZ);
    const uint64_t dring = smem_desc(sb + C::OFF_RING, 16, 1024, kSw128);
    const uint64_t dring_pe = smem_desc(sb + C::OFF_RING, 16, 8 * C::PE_ROW, C::PE_SWZ);
    const uint64_t dpair = smem_desc(sb + C::OFF_RING, C::PBOX, 1024, kSw128);  // Z slab read MN-major
    RingPos rp;
    bool first_o = true;
    // A ring item written by TMA is ordered before the MMAs that read it by its mbarrier
    // alone; tcgen05 fences are needed only where other threads touched Tensor Memory (P).
    auto take = [&](int& slot) -> bool {
      slot = rp.slot;
      const uint32_t ph = rp.phase;
      rp.advance();
      return warp_wait_fast(&r_full[slot], ph, p.wait_ns, abort_flag);
    };
    auto chunk = [&](int u, int j) -> bool {
      if (u == 0 && !warp_wait(&q_box[j], 0, p.wait_ns, abort_flag)) return false;  // Q' box j (TMA)
      int slot;
      if (!take(slot)) return false;
      const uint32_t d_s = tmem + C::TM_S + (u & 1) * TK;
      const uint64_t so = (uint64_t)((slot * C::SLOT) >> 4);
      if (j < C::NBL) {
        const uint64_t qa = dq0 + (uint64_t)((j * C::Q_BOX) >> 4);
        const uint64_t kb = dring + so;
        const uint32_t acc0 = j > 0 ? 1u : 0u;
        if (leader) {
          tc_mma_ss(d_s, qa, kb, idS, acc0);
          tc_mma_ss(d_s, qa + 2, kb + 2, idS, 1u);
          tc_mma_ss(d_s, qa + 4, kb + 4, idS, 1u);
          tc_mma_ss(d_s, qa + 6, kb + 6, idS, 1u);
          tc_commit(&r_empty[slot]);
        }
      } else {
        const uint64_t kb = dring_pe + so;
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < P / 16; ++kk) tc_mma_ss(d_s, dqpe + 2 * kk, kb + 2 * kk, idS, 1u);
          tc_commit(&r_empty[slot]);
        }
      }
      __syncwarp();
      return true;
    };
    auto pair = [&](int v, int q) -> bool {
      if (q == 0) {
        if (!warp_wait(p_full, v & 1, p.wait_ns, abort_flag)) return false;
        tc_fence_after();  // P was written to Tensor Memory by the softmax warps
      }
      int slot;
      if (!take(slot)) return false;
      const int nsl = tile_slabs(v);
      const int key_q = kstart + v * TK + q * PAIR;
      const int first_bad = L - key_q;  // rows of the item at or past the sequence end
      const uint32_t base = C::OFF_RING + slot * C::SLOT;
      if (first_bad < PAIR) {
        const int nrow = PAIR - first_bad;
        for (int idx = lane; idx < nrow * (C::KLH / 64) * 8; idx += 32) {
          const int rr = first_bad + idx / ((C::KLH / 64) * 8);
          const int rem = idx % ((C::KLH / 64) * 8);
          *reinterpret_cast<uint4*>(smem + base + (rem / 8) * C::PBOX + rr * 128 + (rem % 8) * 16) =
              make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      const uint64_t zb = dpair + (uint64_t)((slot * C::SLOT) >> 4);
      const uint32_t a0 = tmem + C::TM_S + (v & 1) * TK + 2 * q * (SLAB / 2);
      const uint32_t acc0 = first_o ? 0u : 1u;
      if (leader) {
        tc_mma_ts(tmem, a0, zb, idO, acc0);
        if (2 * q + 1 < nsl) tc_mma_ts(tmem, a0 + SLAB / 2, zb + (uint64_t)((SLAB * 128) >> 4), idO, 1u);
        tc_commit(&r_empty[slot]);
      }
      first_o = false;
      __syncwarp();
      return true;
    };
    for (int u = 0; ok && u <= ntiles; ++u) {
      ok = walk_iteration<C::NCH, C::J0>(u, ntiles, tile_pairs(u - 1), chunk, pair);
      if (ok && leader) tc_commit(u < ntiles ? &s_ready[u & 1] : o_final);
      __syncwarp();
    }
    if (lane == 0 && !ok && !*abort_flag) fail();
    // every issued tcgen05 operation has finished before TMEM is released
    if (leader) {
      tc_commit(fin_bar);
      mbar_wait(fin_bar, 0, kTeardownNs, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax + epilogue (warps 2-9)
    const int q = warp & 3;            // TMEM lane quadrant this warp may access
    const int ch = (warp - 2) >> 2;    // key half of each tile (and output column half) of this warp
    const int r = q * 32 + lane;
    const int row_in_seq = mt * BMROWS + r;
    const bool row_ok = row_in_seq < p.rows;
    const int lim = row_ok ? min(kend, L - p.s + (row_in_seq % p.s) + 1) : 0;  // exclusive key limit
    const uint32_t t_lane = tmem + ((uint32_t)(q * 32) << 16);
    constexpr int KH = TK / 2;         // keys per warp per tile
    constexpr int OCW = C::KLH / 2;    // O columns per warp (rescale, epilogue)
    float m_ref = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      // S(t) in TMEM; O MMAs of tile t-1 are complete too (issued before this commit).
      // Both warps of a quadrant meet at the exchange below on every tile, whatever
      // happened to their waits, so they leave the loop together (no barrier is orphaned).
      const bool okw = warp_wait(&s_ready[t & 1], (t >> 1) & 1, p.wait_ns, abort_flag);
      const int kb = kstart + t * TK + ch * KH;  // first key of this warp's half
      const uint32_t sbuf = t_lane + C::TM_S + (t & 1) * TK;
      float x[KH];
      float mx = -INFINITY;
      if (okw) {
        tc_fence_after();
        uint32_t sv[32];
        tmem_ld32(sbuf + ch * KH, sv);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; ++c) x[c] = __uint_as_float(sv[c]) * p.scale_log2;
        tmem_ld32(sbuf + ch * KH + 32, sv);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; ++c) x[32 + c] = __uint_as_float(sv[c]) * p.scale_log2;
        if (kb + KH > lim) {
#pragma unroll
          for (int c = 0; c < KH; ++c)
            if (kb + c >= lim) x[c] = -INFINITY;
        }
        float m8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) m8[e] = x[e];
#pragma unroll
        for (int c = 8; c < KH; ++c) m8[c & 7] = fmaxf(m8[c & 7], x[c]);
        mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                   fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      }
      // row maximum over both key halves (the two warps of this quadrant)
      float* rb = red + (t & 1) * 2 * BMROWS;
      rb[ch * BMROWS + r] = mx;
      if (lane == 0) okf[(t & 1) * 8 + ch * 4 + q] = okw ? 1 : 0;
      named_bar_sync(1 + q, 64);
      mx = fmaxf(mx, rb[(ch ^ 1) * BMROWS + r]);
      if (!okw || !okf[(t & 1) * 8 + (ch ^ 1) * 4 + q]) {
        ok = false;
        break;
      }
      float alpha = 1.f;
      if (mx > m_ref + kRescaleLog2) {
        alpha = fast_exp2(m_ref - mx);  // 0 when nothing was seen yet
        m_ref = mx;
        l_run *= alpha;
      }
      if (t > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
        for (int c0 = 0; c0 < OCW; c0 += 32) {
          uint32_t v[32];
          tmem_ld32(t_lane + ch * OCW + c0, v);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * alpha);
          tmem_st32(t_lane + ch * OCW + c0, v);
        }
      }
      // P (bf16 pairs, key 2c in the low half) over columns [ch*32, ch*32+32) of this S buffer
      const float mneg = m_ref == -INFINITY ? 0.f : -m_ref;  // all keys masked so far: x = -inf -> 0
      float ps[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pk[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const float p0 = fast_exp2(x[2 * e] + mneg);
        const float p1 = fast_exp2(x[2 * e + 1] + mneg);
        ps[e & 3] += p0 + p1;
        pk[e] = pack_bf16(p0, p1);
      }
      tmem_st32(sbuf + ch * (KH / 2), pk);
      l_run += (ps[0] + ps[1]) + (ps[2] + ps[3]);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    if (ok && !warp_wait(o_final, 0, p.wait_ns, abort_flag)) ok = false;
    // row sum over both key halves
    float* lb = red + 2 * BMROWS * ((ntiles) & 1);
    lb[ch * BMROWS + r] = l_run;
    named_bar_sync(1 + q, 64);
    const float l_tot = l_run + lb[(ch ^ 1) * BMROWS + r];
    if (!ok) {
      if (!*abort_flag) fail();
    } else {
      tc_fence_after();
      const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
      const float lse = l_tot > 0.f ? (m_ref + log2f(l_tot)) * kLn2 : -INFINITY;
      const size_t grow = (size_t)qrow0 + r;
      // O / l of this warp's 32 rows x OCW columns is staged in shared memory (the query tile's
      // and ring space: every MMA and copy has completed once o_final fired) and stored as
      // whole row segments. Straight from the TMEM layout (thread = row) every store
      // instruction would touch 32 rows with 16 bytes each. Staged rows are 16-byte units
      // XOR-swizzled by (row & 7), so the column-wise writes and the row-wise reads are
      // free of bank conflicts.
      constexpr int F4 = OCW / 4;     // 16-byte units per staged row
      constexpr int ROWB = OCW * 4;   // bytes per staged row
      constexpr int RPI = 32 / F4;    // rows per store instruction
      static_assert(F4 >= 8 && F4 <= 32 && NSMW * 32 * ROWB <= C::OFF_RED, "epilogue staging");
      uint8_t* stg = smem + (warp - 2) * 32 * ROWB;
#pragma unroll 1
      for (int c0 = 0; c0 < OCW; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(t_lane + ch * OCW + c0, v);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 8; ++e)
          *reinterpret_cast<float4*>(stg + lane * ROWB + (((c0 / 4 + e) ^ (lane & 7)) * 16)) =
              make_float4(__uint_as_float(v[4 * e + 0]) * inv, __uint_as_float(v[4 * e + 1]) * inv,
                          __uint_as_float(v[4 * e + 2]) * inv, __uint_as_float(v[4 * e + 3]) * inv);
      }
      __syncwarp();
      const int jl = lane % F4;
#pragma unroll 4
      for (int rr = lane / F4; rr < 32; rr += RPI) {
        const int rs = q * 32 + rr;  // row within the tile
        if (mt * BMROWS + rs >= p.rows) continue;
        const float4 x = *reinterpret_cast<const float4*>(stg + rr * ROWB + ((jl ^ (rr & 7)) * 16));
        const size_t g = (size_t)qrow0 + rs;
        const int col = lh * C::KLH + ch * OCW + jl * 4;
        if (p.nsplit == 1)
          *reinterpret_cast<uint2*>(p.o_lat + g * KL + col) = make_uint2(pack_bf16(x.x, x.y), pack_bf16(x.z, x.w));
        else
          *reinterpret_cast<float4*>(p.ws_o + (g * p.nsplit + split) * KL + col) = x;
      }
      if (row_ok && lh == 0 && ch == 0) {
        if (p.nsplit == 1) {
          if (p.lse) p.lse[grow] = lse;
        } else {
          p.ws_lse[grow * p.nsplit + split] = lse;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(*tmem_slot, C::TM_COLS);
  }
}

// ---------------------------------------------------------------------------
// host side: tensor maps and launch

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

CUtensorMapSwizzle swizzle_for(int row_bytes) {
  return row_bytes >= 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                          : (row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
}

// 2-D bf16 map over a [rows, cols] row-major matrix with boxes [box_rows, box_cols]
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows, uint32_t box_cols) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for((int)box_cols * 2), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int KL, int P>
cudaError_t launch_kl(const MlaLaunch& a, cudaStream_t stream) {
  using C = MlaCfg<KL, P>;
  static std::atomic<unsigned long long> smem_limit_set{0};
  if (cudaError_t e = ensure_smem_limit(mla_latent_kernel<KL, P>, C::SMEM, smem_limit_set)) return e;
  const uint64_t qrows = (uint64_t)a.b * a.h * a.s;
  const uint64_t krows = a.paged ? (uint64_t)a.num_pages * 64 : (uint64_t)a.b * a.capacity;
  CUtensorMap tqz, tqpe, tz64, tkpe64, tz32;
  if (!make_map(&tqz, a.qz, qrows, KL, BMROWS, 64) || !make_map(&tqpe, a.q_pe, qrows, P, BMROWS, P) ||
      !make_map(&tz64, a.z, krows, KL, 64, 64) || !make_map(&tkpe64, a.k_pe, krows, P, 64, P) ||
      !make_map(&tz32, a.z, krows, KL, PAIR, 64))
    return cudaErrorInvalidValue;
  MlaParams p;
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
  p.ws_o = a.ws_o;
  p.ws_lse = a.ws_lse;
  p.err = a.err;
  p.wait_ns = a.wait_ns;
  p.test_timeout = a.test_timeout;
  const int mtiles = (p.rows + BMROWS - 1) / BMROWS;
  // programmatic dependent launch: the set-up overlaps the previous kernel (see pdl_wait)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C::NH * mtiles, a.nsplit, a.b);
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, mla_latent_kernel<KL, P>, tqz, tqpe, tz64, tkpe64, tz32, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

int mla_latent_parts(int k) { return k >= 512 ? 2 : 1; }
int mla_tile_keys() { return TK; }
bool mla_supported(int k, int p) { return (k == 512 && p == 64) || (k == 64 && p == 16); }

cudaError_t launch_mla_latent(const MlaLaunch& a, cudaStream_t stream) {
  if (a.k == 512 && a.p == 64) return launch_kl<512, 64>(a, stream);
  if (a.k == 64 && a.p == 16) return launch_kl<64, 16>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace decattn
