// Grouped-head attention for many query rows per KV head (prefill-sized s) on the
// tensor cores (sm_103a).
//
// "Mla Analysis" skill page, Regime Selection (the Prefill row: plain attention over
// decompressed keys wins at large s) and Cost Models — FlashAttention; the grouped-head
// rows of the summary table in "Why MLA and MTP Fight Each Other". The same computation
// as the split-KV decode kernel (row = head_in_group * s + token, a causal window
// aligned to the end), for KV heads with at least 64 query rows, where the mma.sync
// kernel's 16-row tiles re-stream the cache once per row block and run out of math.
//
// One CTA takes 128 query rows of one (sequence, KV head) and every key they see, or a
// piece of those keys:
//  * Q [128 rows x DK] comes by TMA through the K ring's first two slots and is moved into
//    Tensor Memory by the softmax warps (lane = row, two bf16 per column), where it stays
//    as the A operand of the score MMAs; shared memory is then all K and V: 64-key tiles
//    in 3 K + 4 V slots (DK = DV = 256), 4 + 8 (192 / 128) or 7 + 7 (128 / 128).
//  * One thread issues tcgen05.mma: S = Q K^T (M = 128, N = 64, A from Tensor Memory)
//    into one of two TMEM buffers, and O += P V (M = 128, N = DV) into a TMEM
//    accumulator, the P V of tile t-1 issued after the S of tile t so that the softmax of
//    tile t overlaps it.
//  * Four softmax warps (thread = row) read S from TMEM, keep a lazy reference maximum
//    (moved only past 2^8; the O row is then rescaled in TMEM once the previous tile's
//    P V has completed), write P as bf16 back into Tensor Memory over its own S columns
//    (the P V takes A from there), and at the end scale O by 1/l and store bf16 rows and
//    the LSE.
//  * K and V have rings of their own, fed by two producer warps: a K slot is free once
//    its score MMA completes, a V slot once its P V has, so the K stream runs ahead of
//    the V stream and more of both is in flight than a shared K+V stage allows.
// Every wait is bounded; a wait that runs out sets the error word and the CTA winds
// down (its copies and MMAs waited for, TMEM freed). V rows past the sequence end are
// zeroed before the MMA reads them (their P is 0, but 0 * NaN is NaN).
//
// Work split. Either a fixed chunk count planned on the host from the longest sequence
// (CTA (rb + nrb * split, KV head, sequence)), or, when the work items (sequence, KV head,
// row block) are fewer than the CTAs of one wave, a balanced split planned on the device
// from the actual lengths: with T key tiles over all items and a grid of C CTAs, every
// item is cut into ceil(tiles / W) near-equal pieces, W = ceil(T / (C - items)), so that
// the pieces fit one wave and none is longer than W tiles. A piece that is a whole item
// writes final rows; the pieces of a cut item write fp32 partial records (record = CTA
// index) merged by the balanced combine.
#include <cstring>

#include "common.cuh"
#include "internal.h"

namespace decattn {

namespace {

constexpr int PM = 128;          // query rows per CTA (MMA M)
constexpr int PK = 64;           // keys per tile (S MMA N)
constexpr int PNS_MAX = 8;       // slots of either ring at most
constexpr int PCH = PK * 128;    // one [64 keys x 64 values] bf16 chunk, 128-byte rows
constexpr int PQCH = PM * 128;   // one [128 rows x 64 values] chunk of Q or P
// warp 0 K (and Q) loads, 1 MMA, 2-5 softmax / epilogue, 6 V loads; FP8: warps 7-10 widen
// the landed K bytes to f16, warps 11-14 the V bytes
constexpr int kPWarpV = 6, kPWarpC0 = 7, kPNCW = 4;
__host__ __device__ constexpr int pf_threads(bool fp8) { return fp8 ? 32 * (7 + 2 * kPNCW) : 224; }
constexpr float kPLog2e = 1.4426950408889634f;
constexpr float kPLn2 = 0.6931471805599453f;
constexpr float kPRescale = 8.f;
constexpr unsigned long long kPTeardownNs = 1000000000ull;

template <int DK, int DV, bool FP8>
struct PfCfg {
  static constexpr int KCH = DK / 64, VCH = DV / 64;
  static constexpr int KT = KCH * PCH, VT = VCH * PCH;  // one 64-key K / V tile (16-bit values)
  // Separate K and V rings: a K slot is free once its score MMA completes, a V slot only
  // once the P V that reads it has. bf16: half the shared memory goes to K (the query lap
  // takes its first two slots), the rest to V. FP8: E4M3 tiles land by TMA in rings of
  // their own (LK / LV bytes a tile) and are widened to f16 into the K and V rings.
  static constexpr int BUDGET = 232448 - 1024 - 1024;  // barriers + slots, alignment slack
  // FP8: the query lap lands in the V ring (free until the first P V), so the K ring is
  // two or three slots and the landing rings take the rest.
  static constexpr int LK = FP8 ? PK * DK : 0, LV = FP8 ? PK * DV : 0;
  static constexpr int NLK = FP8 ? (DK == 256 ? 3 : 7) : 0, NLV = NLK;
  static constexpr int NK_FIT = (BUDGET / 2) / KT;
  static constexpr int NK = FP8 ? (DK == 256 ? 2 : 3) : (NK_FIT < PNS_MAX ? NK_FIT : PNS_MAX);
  static constexpr int NV_FIT = (BUDGET - NK * KT) / VT;
  static constexpr int NV = FP8 ? (DK == 256 ? 2 : 4) : (NV_FIT < PNS_MAX ? NV_FIT : PNS_MAX);
  static constexpr int QBYTES = KCH * PQCH;                      // Q [128 rows x DK] bf16
  static constexpr int QS = FP8 ? 0 : (QBYTES + KT - 1) / KT;    // K slots the query lap covers
  static constexpr int QSV = FP8 ? (QBYTES + VT - 1) / VT : 0;   // V slots the query lap covers
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + NK * KT;
  static constexpr int OFF_LK = OFF_V + NV * VT;
  static constexpr int OFF_LV = OFF_LK + NLK * LK;
  static constexpr int OFF_BAR = OFF_LV + NLV * LV;
  static constexpr int SMEM = OFF_BAR + 1024 + 1024;
  // Tensor Memory: two S buffers (columns 0 and PK; P is written over the first PK / 2
  // columns of its own S), O (2 PK), Q (2 PK + DV, DK / 2 columns)
  static constexpr int OCOL = 2 * PK, QCOL = 2 * PK + DV;
  static constexpr int TMEM_COLS = 512;
  static_assert(DK % 64 == 0 && DV % 64 == 0 && DV <= 256, "widths");
  static_assert(!FP8 || (DK == DV && (DK == 128 || DK == 256)), "FP8 widths");
  static_assert(QCOL + DK / 2 <= TMEM_COLS, "tensor memory");
  static_assert(NK >= 2 && NV >= 2 && QS < NK && QSV <= NV && QBYTES <= (FP8 ? NV * VT : NK * KT) &&
                    OFF_V % 1024 == 0 && KT % 1024 == 0,
                "rings");
  static_assert(SMEM <= 232448, "shared memory");
};

// barriers
enum { F_QREADY = 0, F_KFULL = 1, F_KEMPTY = F_KFULL + PNS_MAX, F_VFULL = F_KEMPTY + PNS_MAX,
       F_VEMPTY = F_VFULL + PNS_MAX, F_SFULL = F_VEMPTY + PNS_MAX, F_PFULL = F_SFULL + 2, F_PVDONE = F_PFULL + 2,
       F_OFINAL = F_PVDONE + 2, F_FIN = F_OFINAL + 1, F_TEST = F_FIN + 1,
       F_LKFULL = F_TEST + 1, F_LKEMPTY = F_LKFULL + PNS_MAX, F_LVFULL = F_LKEMPTY + PNS_MAX,
       F_LVEMPTY = F_LVFULL + PNS_MAX, F_QLAND = F_LVEMPTY + PNS_MAX, F_COUNT = F_QLAND + 1 };
static_assert(F_COUNT * 8 + 8 <= 1024, "barrier region");
constexpr int kPBarQ = 1;  // named barrier of the four softmax warps
constexpr unsigned long long kPTestWaitNs = 1000000ull;  // forced-timeout test: 1 ms

struct PfParams {
  const __nv_bfloat16* q;
  __nv_bfloat16* out;
  float* lse;
  const int32_t* seqlens;
  const int32_t* block_table;
  int max_pages, paged, capacity, num_pages;
  int b, s, hq, hkv, G, R, nrb;
  int nsplit, chunk;  // context split: CTA x covers keys [split * chunk, (split + 1) * chunk)
  float* ws_o;        // nsplit > 1: fp32 partials [b*Hq*s rows][nsplit][DV] (normalised O);
                      // balanced: records [grid][PM rows][DV]
  float* ws_lse;      // and their LSEs [rows][nsplit] / [grid][PM]
  int balanced;       // nonzero: the device-planned balanced split over a 1-D grid
  int* meta;          // balanced: [work items][2] {first record, count}
  float scale_log2;  // softmax scale x log2(e) (FP8: x k_scale)
  float v_scale;     // FP8: dequantisation scale of V (1 for bf16)
  unsigned* err;
  unsigned long long wait_ns;
  int test_timeout;  // nonzero: the first softmax wait also waits on a barrier nothing signals
};

// all lanes of a warp wait (bounded); true only if every lane saw the phase complete
__device__ __forceinline__ bool pf_wait(uint64_t* bar, uint32_t parity, unsigned long long ns, volatile int* abort_flag) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, ns, abort_flag));
}

// keys seen by row block rb of a sequence of L keys: the widest causal window among the
// block's rows (row = head_in_group * s + token)
__device__ __forceinline__ int pf_kwin(const PfParams& p, int L, int rb) {
  const int r0 = rb * PM, r1 = min(p.R, r0 + PM);
  const int maxtok = (r1 - r0 >= p.s || r0 / p.s != (r1 - 1) / p.s) ? p.s - 1 : (r1 - 1) % p.s;
  return L >= p.s ? min(L, L - p.s + maxtok + 1) : (L > 0 ? L : 0);
}

// this CTA's work: item (sequence bi, KV head g, row block rb) and key range; n = pieces
// of the item (1: final rows), first = its first record; valid = false: no work
struct PfPiece {
  int bi, g, rb, kstart, kend, n, first;
  long long item;
  bool valid;
};
__device__ PfPiece pf_piece(const PfParams& p) {
  PfPiece w{};
  if (!p.balanced) {
    w.rb = blockIdx.x % p.nrb;
    const int split = blockIdx.x / p.nrb;
    w.g = blockIdx.y;
    w.bi = blockIdx.z;
    w.kstart = split * p.chunk;
    w.kend = min(pf_kwin(p, p.seqlens[w.bi], w.rb), w.kstart + p.chunk);
    w.n = p.nsplit;
    w.first = split;
    w.valid = true;
    return w;
  }
  const long long items = (long long)p.b * p.hkv * p.nrb;
  auto tiles_of = [&](long long it) -> long long {
    const int bi = (int)(it / ((long long)p.hkv * p.nrb));
    return (pf_kwin(p, __ldg(p.seqlens + bi), (int)(it % p.nrb)) + PK - 1) / PK;
  };
  long long total = 0;
  for (long long it = 0; it < items; ++it) total += tiles_of(it);
  const long long spare = (long long)gridDim.x - items;  // > 0 (the host checks)
  const long long W = spare > 0 ? max(1ll, (total + spare - 1) / spare) : max(1ll, total);
  const long long c = blockIdx.x;
  long long prefix = 0;
  for (long long it = 0; it < items; ++it) {
    const long long tiles = tiles_of(it);
    const long long n = (tiles + W - 1) / W;
    if (c < prefix + n) {
      const long long j = c - prefix;
      const int L = __ldg(p.seqlens + (int)(it / ((long long)p.hkv * p.nrb)));
      w.item = it;
      w.rb = (int)(it % p.nrb);
      w.g = (int)((it / p.nrb) % p.hkv);
      w.bi = (int)(it / ((long long)p.hkv * p.nrb));
      w.kstart = (int)((j * tiles / n) * PK);
      w.kend = min(pf_kwin(p, L, w.rb), (int)(((j + 1) * tiles / n) * PK));
      w.n = (int)n;
      w.first = (int)prefix;
      w.valid = true;
      return w;
    }
    prefix += n;
  }
  w.valid = false;  // beyond the last piece: nothing to do
  return w;
}

// Widen one landed tile of 64 rows x W E4M3 bytes ([row][W]) to f16 in the chunk-major,
// 128-byte swizzled layout of the K / V rings ([W/64 chunks][64 rows][64 values]); the
// threads of one group of kPNCW warps share the work, 16 bytes (16 values) each.
template <int W>
__device__ __forceinline__ void widen_e4m3_tile(const uint8_t* land, uint8_t* dst, int tid) {
  constexpr int UPR = W / 16;  // 16-byte units of a landed row
#pragma unroll 4
  for (int idx = tid; idx < PK * UPR; idx += 32 * kPNCW) {
    const int row = idx / UPR, v = idx % UPR;
    const uint4 x = *reinterpret_cast<const uint4*>(land + row * W + v * 16);
    uint32_t lo[4], hi[4];
    e4m3x4_to_f16x2x2(x.x, lo[0], hi[0]);
    e4m3x4_to_f16x2x2(x.y, lo[1], hi[1]);
    e4m3x4_to_f16x2x2(x.z, lo[2], hi[2]);
    e4m3x4_to_f16x2x2(x.w, lo[3], hi[3]);
    // values 16v .. 16v+15: chunk v / 4, 16-byte units 2 (v % 4) and the next
    const int u0 = (v & 3) * 2;
    uint8_t* rowp = dst + (v >> 2) * PCH + row * 128;
    *reinterpret_cast<uint4*>(rowp + ((u0 ^ (row & 7)) << 4)) = make_uint4(lo[0], hi[0], lo[1], hi[1]);
    *reinterpret_cast<uint4*>(rowp + (((u0 + 1) ^ (row & 7)) << 4)) = make_uint4(lo[2], hi[2], lo[3], hi[3]);
  }
}

template <int DK, int DV, bool FP8>
__global__ void __launch_bounds__(pf_threads(FP8), 1)
    gqa_prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, PfParams p) {
  using C = PfCfg<DK, DV, FP8>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the 128-byte swizzle wants 1024-byte aligned tiles: round the base up (slack reserved)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + F_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + F_COUNT) + 1;

  if (threadIdx.x == 0) {
    mbar_init(&bars[F_QREADY], 1);
    mbar_init(&bars[F_QLAND], 1);
    // FP8: the K / V rings are filled by the widening warps (one arrival each), the
    // landing rings emptied by them
    for (int i = 0; i < C::NK; ++i) {
      mbar_init(&bars[F_KFULL + i], FP8 ? kPNCW : 1);
      mbar_init(&bars[F_KEMPTY + i], 1);
    }
    for (int i = 0; i < C::NV; ++i) {
      mbar_init(&bars[F_VFULL + i], FP8 ? kPNCW : 1);
      mbar_init(&bars[F_VEMPTY + i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[F_SFULL + i], 1);
      mbar_init(&bars[F_PFULL + i], 4);
      mbar_init(&bars[F_PVDONE + i], 1);
    }
    for (int i = 0; i < C::NLK; ++i) {
      mbar_init(&bars[F_LKFULL + i], 1);
      mbar_init(&bars[F_LKEMPTY + i], kPNCW);
    }
    for (int i = 0; i < C::NLV; ++i) {
      mbar_init(&bars[F_LVFULL + i], 1);
      mbar_init(&bars[F_LVEMPTY + i], kPNCW);
    }
    mbar_init(&bars[F_OFINAL], 1);
    mbar_init(&bars[F_FIN], 1);
    mbar_init(&bars[F_TEST], 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;  // S buffers at columns 0 and PK, O at 2 PK, Q after O
  auto fail = [&]() {
    raise_error(p.err, kErrWaitTimeout);
    *abort_flag = 1;
  };
  pdl_wait();  // queries, cache and lengths may come from the previous kernel in the stream
  pdl_trigger();

  const PfPiece w = pf_piece(p);
  const int rb = w.rb, g = w.g, bi = w.bi;
  const int L = w.valid ? p.seqlens[bi] : 0;
  const int r0 = rb * PM;  // first row (within the KV head's R rows) of the block
  const int kstart = w.kstart, kend = w.kend;
  const int ntiles = w.valid && kend > kstart ? (kend - kstart + PK - 1) / PK : 0;
  const int qrow0 = (bi * p.hq + g * p.G) * p.s + r0;  // first flattened [b*hq*s] query row

  // token row of tile t's first key in the cache tensor (a tile is one page)
  auto tile_row = [&](int t) -> int {
    if (p.paged) {
      int page = __ldg(p.block_table + (size_t)bi * p.max_pages + kstart / PK + t);
      if (page < 0 || page >= p.num_pages) {
        raise_error(p.err, kErrBadPage);
        page = 0;  // stay inside the pool; the result is flagged invalid
      }
      return page * PK;
    }
    return bi * p.capacity + kstart + t * PK;
  };

  if (warp == 0) {
    // ------------------------------------------------ TMA producer: the query lap, then K tiles
    if (ntiles > 0 && elect_one()) {
      // the query lap: Q boxes [128 rows x 64] (16 KB each) laid end to end from the K ring's
      // start over its first QS slots; a box completes on the barrier of the slot it starts
      // in, and a slot in which no box starts gets a plain arrival
      if constexpr (FP8) {
        // FP8: the whole lap completes on its own barrier, in the V ring's first QSV slots
        mbar_expect_tx(&bars[F_QLAND], C::QBYTES);
        for (int c = 0; c < C::KCH; ++c) tma_load_2d(sb + C::OFF_V + c * PQCH, &tm_q, c * 64, qrow0, &bars[F_QLAND]);
      } else {
        uint32_t qbytes[C::QS > 0 ? C::QS : 1];
        for (int i = 0; i < C::QS; ++i) qbytes[i] = 0;
        for (int c = 0; c < C::KCH; ++c) qbytes[(c * PQCH) / C::KT] += PQCH;
        for (int i = 0; i < C::QS; ++i) {
          if (qbytes[i])
            mbar_expect_tx(&bars[F_KFULL + i], qbytes[i]);
          else
            mbar_arrive(&bars[F_KFULL + i]);
        }
        for (int c = 0; c < C::KCH; ++c)
          tma_load_2d(sb + C::OFF_K + c * PQCH, &tm_q, c * 64, qrow0, &bars[F_KFULL + (c * PQCH) / C::KT]);
      }
      // K of tile t takes K-ring position u = QS + t: slot u % NK, its (u / NK)-th use. One
      // box per tile ([chunks][64 keys][64 values], chunk-major as the MMAs read it: the
      // TMA engine serves about one box per few hundred cycles per SM whatever its size).
      int last[PNS_MAX];
      for (int i = 0; i < PNS_MAX; ++i) last[i] = i < C::QS ? i : -1;
      int lastl[PNS_MAX];
      for (int i = 0; i < PNS_MAX; ++i) lastl[i] = -1;
      for (int t = 0; t < ntiles; ++t) {
        if constexpr (FP8) {  // E4M3 bytes [64 rows x DK] into landing slot t % NLK
          const int ls = t % C::NLK;
          if (t >= C::NLK && !mbar_wait(&bars[F_LKEMPTY + ls], ((t / C::NLK) - 1) & 1, p.wait_ns, abort_flag)) {
            if (!*abort_flag) fail();
            break;
          }
          mbar_expect_tx(&bars[F_LKFULL + ls], C::LK);
          tma_load_3d(sb + C::OFF_LK + ls * C::LK, &tm_k, 0, g, tile_row(t), &bars[F_LKFULL + ls]);
          lastl[ls] = t;
        } else {
          const int u = C::QS + t, slot = u % C::NK;
          if (u >= C::NK && !mbar_wait(&bars[F_KEMPTY + slot], ((u / C::NK) - 1) & 1, p.wait_ns, abort_flag)) {
            if (!*abort_flag) fail();
            break;
          }
          mbar_expect_tx(&bars[F_KFULL + slot], C::KT);
          tma_load_4d(sb + C::OFF_K + slot * C::KT, &tm_k, 0, tile_row(t), 0, g, &bars[F_KFULL + slot]);
          last[slot] = u;
        }
      }
      // leave no copy in flight (FP8: the query lap's slots here, the landings below)
      for (int i = 0; i < C::NK; ++i)
        if (last[i] >= 0) mbar_wait(&bars[F_KFULL + i], (last[i] / C::NK) & 1, kPTeardownNs, nullptr);
      if constexpr (FP8) {
        for (int i = 0; i < C::NLK; ++i)
          if (lastl[i] >= 0) mbar_wait(&bars[F_LKFULL + i], (lastl[i] / C::NLK) & 1, kPTeardownNs, nullptr);
        mbar_wait(&bars[F_QLAND], 0, kPTeardownNs, nullptr);
      }
    }
    __syncwarp();
  } else if (warp == kPWarpV) {
    // ------------------------------------------------ TMA producer: V tiles (slot t % NV)
    if (ntiles > 0 && elect_one()) {
      int last[PNS_MAX];
      for (int i = 0; i < PNS_MAX; ++i) last[i] = -1;
      constexpr int NR = FP8 ? C::NLV : C::NV;  // FP8: V lands in its own ring first
      for (int t = 0; t < ntiles; ++t) {
        const int slot = t % NR;
        uint64_t* full = &bars[(FP8 ? F_LVFULL : F_VFULL) + slot];
        if (t >= NR && !mbar_wait(&bars[(FP8 ? F_LVEMPTY : F_VEMPTY) + slot], ((t / NR) - 1) & 1, p.wait_ns, abort_flag)) {
          if (!*abort_flag) fail();
          break;
        }
        if constexpr (FP8) {
          mbar_expect_tx(full, C::LV);
          tma_load_3d(sb + C::OFF_LV + slot * C::LV, &tm_v, 0, g, tile_row(t), full);
        } else {
          mbar_expect_tx(full, C::VT);
          tma_load_4d(sb + C::OFF_V + slot * C::VT, &tm_v, 0, tile_row(t), 0, g, full);
        }
        last[slot] = t;
      }
      for (int i = 0; i < NR; ++i)
        if (last[i] >= 0) mbar_wait(&bars[(FP8 ? F_LVFULL : F_VFULL) + i], (last[i] / NR) & 1, kPTeardownNs, nullptr);
    }
    __syncwarp();
  } else if (warp >= kPWarpC0) {  // FP8 instances only (bf16 has 7 warps)
    // ------------------------------------------------ widen landed E4M3 tiles to f16 (K: warps 7-10, V: 11-14)
    // K tile t goes to K-ring position QS + t (after the query lap), V tile t to V-ring
    // slot t % NV; a ring slot is taken once the MMA that read it last has completed, and
    // the landing slot is released once its bytes have been read.
    if constexpr (FP8) {
    const bool isk = warp < kPWarpC0 + kPNCW;
    const int tid = ((warp - kPWarpC0) % kPNCW) * 32 + lane;  // thread within the group
    const int NL = isk ? C::NLK : C::NLV;
    bool ok = true;
    for (int t = 0; ok && t < ntiles; ++t) {
      const int ls = t % NL;
      const int u = isk ? C::QS + t : C::QSV + t;  // ring position after the query lap
      const int NR = isk ? C::NK : C::NV;
      const int rs = u % NR;
      if (!pf_wait(&bars[(isk ? F_LKFULL : F_LVFULL) + ls], (t / NL) & 1, p.wait_ns, abort_flag) ||
          (u >= NR && !pf_wait(&bars[(isk ? F_KEMPTY : F_VEMPTY) + rs], ((u / NR) - 1) & 1, p.wait_ns, abort_flag))) {
        ok = false;
        break;
      }
      if (isk)
        widen_e4m3_tile<DK>(smem + C::OFF_LK + ls * C::LK, smem + C::OFF_K + rs * C::KT, tid);
      else
        widen_e4m3_tile<DV>(smem + C::OFF_LV + ls * C::LV, smem + C::OFF_V + rs * C::VT, tid);
      fence_proxy_async_smem();  // the MMAs and the next landing copy (async proxy) come after these accesses
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars[(isk ? F_KFULL : F_VFULL) + rs]);
        mbar_arrive(&bars[(isk ? F_LKEMPTY : F_LVEMPTY) + ls]);
      }
    }
    if (!ok && lane == 0 && !*abort_flag) fail();
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (the whole warp waits; one lane issues)
    const bool leader = elect_one();
    // bf16 operands, or f16 (FP8 cache widened exactly to f16; Q and P in f16 too)
    constexpr uint32_t idS = FP8 ? idesc_f16_f32(PM, PK, false, false) : idesc_bf16_f32(PM, PK, false, false);
    constexpr uint32_t idO = FP8 ? idesc_f16_f32(PM, DV, false, true) : idesc_bf16_f32(PM, DV, false, true);
    const uint64_t dk = smem_desc(sb + C::OFF_K, 16, 1024, kSw128);
    const uint64_t dv = smem_desc(sb + C::OFF_V, PCH, 1024, kSw128);  // chunk stride 8 KB
    bool ok = ntiles == 0 || pf_wait(&bars[F_QREADY], 0, p.wait_ns, abort_flag);
    tc_fence_after();  // Q was written to Tensor Memory by the softmax warps
    // O += P(u) V(u), P(u) from Tensor Memory (over S buffer u & 1); the tail of the last
    // tile's V rows is zeroed first
    auto o_mma = [&](int u) -> bool {
      // V of tile u sits at V-ring position QSV + u (FP8: the query lap took the first QSV
      // positions without completing their full barriers, so those slots' completions lag
      // one lap)
      const int pv = C::QSV + u;
      const int pb = u & 1, slot = pv % C::NV;
      const int vph = (pv / C::NV - (slot < C::QSV ? 1 : 0)) & 1;
      if (!pf_wait(&bars[F_PFULL + pb], (u >> 1) & 1, p.wait_ns, abort_flag) ||
          !pf_wait(&bars[F_VFULL + slot], vph, p.wait_ns, abort_flag))
        return false;
      const int nvalid = kend - (kstart + u * PK);
      if (nvalid < PK) {
        uint8_t* vt = smem + C::OFF_V + slot * C::VT;
        for (int idx = lane; idx < (PK - nvalid) * C::VCH * 8; idx += 32) {
          const int row = nvalid + idx / (C::VCH * 8), rem = idx % (C::VCH * 8);
          *reinterpret_cast<uint4*>(vt + (rem / 8) * PCH + row * 128 + (rem % 8) * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      tc_fence_after();
      if (leader) {
        const uint64_t b0 = dv + (uint64_t)((slot * C::VT) >> 4);
#pragma unroll
        for (int kk = 0; kk < PK / 16; ++kk)
          tc_mma_ts(tmem + C::OCOL, tmem + pb * PK + kk * 8, b0 + (uint64_t)((kk * 16 * 128) >> 4), idO,
                    (u > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&bars[F_VEMPTY + slot]);  // the V slot is free
        tc_commit(&bars[F_PVDONE + pb]);    // S/P buffer pb is free; O holds tiles <= u
      }
      __syncwarp();
      return true;
    };
    for (int t = 0; ok && t < ntiles; ++t) {
      const int u = C::QS + t, slot = u % C::NK, sbuf = t & 1;
      // K of tile t landed; S buffer sbuf (P of tile t - 2) has been read by its P V
      if (!pf_wait(&bars[F_KFULL + slot], (u / C::NK) & 1, p.wait_ns, abort_flag) ||
          (t >= 2 && !pf_wait(&bars[F_PVDONE + sbuf], ((t >> 1) - 1) & 1, p.wait_ns, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (leader) {
        const uint64_t b0 = dk + (uint64_t)((slot * C::KT) >> 4);
#pragma unroll
        for (int kk = 0; kk < DK / 16; ++kk)
          tc_mma_ts(tmem + sbuf * PK, tmem + C::QCOL + kk * 8, b0 + (uint64_t)(((kk / 4) * PCH + (kk % 4) * 32) >> 4),
                    idS, kk > 0 ? 1u : 0u);
        tc_commit(&bars[F_KEMPTY + slot]);  // the K slot is free once these MMAs complete
        tc_commit(&bars[F_SFULL + sbuf]);
      }
      __syncwarp();
      if (t >= 1 && !o_mma(t - 1)) ok = false;
    }
    if (ok && ntiles > 0) ok = o_mma(ntiles - 1);
    if (leader) {
      if (ok && ntiles > 0) tc_commit(&bars[F_OFINAL]);
      if (!ok && !*abort_flag) fail();
      // every MMA issued has completed before Tensor Memory is freed
      tc_commit(&bars[F_FIN]);
      mbar_wait(&bars[F_FIN], 0, kPTeardownNs, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ softmax (thread = row = TMEM lane), then the epilogue
    const int q = warp & 3;            // TMEM lane quadrant this warp may access
    const int r = q * 32 + lane;       // row within the block
    const int rg = r0 + r;             // row within the KV head
    const bool row_ok = rg < p.R;
    const int tok = rg % p.s;
    const int lim = row_ok ? (L >= p.s ? min(kend, L - p.s + tok + 1) : kend) : 0;  // exclusive key limit
    const uint32_t t_lane = tmem + ((uint32_t)(q * 32) << 16);
    float m_ref = -INFINITY, l_run = 0.f;
    bool ok = ntiles > 0;
    if (ntiles > 0) {
      // Q row r into Tensor Memory (A operand of the score MMAs: lane = row, two bf16 per
      // column, even index low); chunk j of the query lap is [128 rows x 64] with 128-byte
      // swizzled rows. Then the query lap's ring slots go back to the producer.
      bool okq = true;
      if constexpr (FP8)
        okq = pf_wait(&bars[F_QLAND], 0, p.wait_ns, abort_flag);
      else
        for (int i = 0; i < C::QS; ++i) okq = okq && pf_wait(&bars[F_KFULL + i], 0, p.wait_ns, abort_flag);
      if (okq) {
#pragma unroll 1
        for (int j = 0; j < C::KCH; ++j) {
          const uint8_t* bx = smem + (FP8 ? C::OFF_V : C::OFF_K) + j * PQCH + r * 128;
          uint32_t v[32];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint4 x = *reinterpret_cast<const uint4*>(bx + ((u ^ (r & 7)) << 4));
            v[4 * u] = x.x;
            v[4 * u + 1] = x.y;
            v[4 * u + 2] = x.z;
            v[4 * u + 3] = x.w;
          }
          if constexpr (FP8) {  // f16 queries for the f16 MMAs (range 2^-14 .. 65504)
#pragma unroll
            for (int c = 0; c < 32; ++c) v[c] = pack_f16(bf16_lo(v[c]), bf16_hi(v[c]));
          }
          tmem_st32(t_lane + C::QCOL + j * 32, v);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      ok = named_bar_and(kPBarQ, 128, okq && !*abort_flag);
      if (threadIdx.x == 64) {
        if (ok) {
          for (int i = 0; i < C::QS; ++i) mbar_arrive(&bars[F_KEMPTY + i]);
          for (int i = 0; i < C::QSV; ++i) mbar_arrive(&bars[F_VEMPTY + i]);
          mbar_arrive(&bars[F_QREADY]);
        } else if (!*abort_flag) {
          fail();
        }
      }
    }
    for (int t = 0; ok && t < ntiles; ++t) {
      const int sbuf = t & 1;
      if (!pf_wait(&bars[F_SFULL + sbuf], (t >> 1) & 1, p.wait_ns, abort_flag) ||
          (t == 0 && p.test_timeout && !pf_wait(&bars[F_TEST], 0, kPTestWaitNs, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      float x[PK];
      {
        uint32_t v[32];
        tmem_ld32(t_lane + sbuf * PK, v);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; ++c) x[c] = __uint_as_float(v[c]) * p.scale_log2;
        tmem_ld32(t_lane + sbuf * PK + 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; ++c) x[32 + c] = __uint_as_float(v[c]) * p.scale_log2;
      }
      const int kb = kstart + t * PK;
      if (kb + PK > lim) {
#pragma unroll
        for (int c = 0; c < PK; ++c)
          if (kb + c >= lim) x[c] = -INFINITY;
      }
      float mx = x[0];
#pragma unroll
      for (int c = 1; c < PK; ++c) mx = fmaxf(mx, x[c]);
      // lazy reference maximum: moved only past 2^8; O (tiles < t, once their P V is done)
      // is then rescaled in TMEM row by row (the whole warp takes part in the loads)
      float alpha = 1.f;
      const bool move = mx > m_ref + kPRescale;
      if (move) alpha = fast_exp2(m_ref - mx);  // 0 while nothing was seen yet
      if (__any_sync(0xffffffffu, move && m_ref != -INFINITY) && t >= 1) {
        if (!pf_wait(&bars[F_PVDONE + ((t - 1) & 1)], ((t - 1) >> 1) & 1, p.wait_ns, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int c0 = 0; c0 < DV; c0 += 32) {
          uint32_t v[32];
          tmem_ld32(t_lane + C::OCOL + c0, v);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * alpha);
          tmem_st32(t_lane + C::OCOL + c0, v);
        }
        tmem_st_wait();
      }
      if (move) {
        m_ref = mx;
        l_run *= alpha;
      }
      const float mneg = m_ref == -INFINITY ? 0.f : -m_ref;  // all keys masked so far: x = -inf -> 0
      uint32_t pk[PK / 2];
      float ps = 0.f;
#pragma unroll
      for (int e = 0; e < PK / 2; ++e) {
        const float p0 = fast_exp2(x[2 * e] + mneg), p1 = fast_exp2(x[2 * e + 1] + mneg);
        ps += p0 + p1;
        pk[e] = FP8 ? pack_f16(p0, p1) : pack_bf16(p0, p1);
      }
      l_run += ps;
      // P row r into Tensor Memory over the first PK / 2 columns of its own S buffer (the A
      // operand of the P V: lane = row, two bf16 per column, even key low); S is in x[]
      tmem_st32(t_lane + sbuf * PK, pk);
      tmem_st_wait();
      tc_fence_before();  // P and the rescale's TMEM stores come before the P V
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[F_PFULL + sbuf]);
    }
    if (ok && ntiles > 0) ok = pf_wait(&bars[F_OFINAL], 0, p.wait_ns, abort_flag);
    if (!ok && ntiles > 0) {
      if (lane == 0 && !*abort_flag) fail();
    } else if (w.valid) {
      // final rows when the item is whole (one piece or no split), else a partial: fp32
      // normalised O and its LSE, by split (fixed chunks) or in record blockIdx.x (balanced)
      const bool whole = w.n <= 1;
      float* part_o = nullptr;
      float* part_l = nullptr;
      tc_fence_after();
      const float inv = l_run > 0.f ? p.v_scale / l_run : 0.f;  // FP8: V's dequantisation scale too
      const float lse_val = l_run > 0.f ? (m_ref + log2f(l_run)) * kPLn2 : -INFINITY;
      const int j = g * p.G + rg / p.s;
      const size_t rowflat = ((size_t)bi * p.hq + j) * p.s + tok;
      if (!whole) {
        const size_t rec = p.balanced ? ((size_t)blockIdx.x * PM + r) : (rowflat * p.nsplit + w.first);
        part_o = p.ws_o + rec * DV;
        part_l = p.ws_lse + rec;
        if (p.balanced && w.kstart == 0 && threadIdx.x == 64) {  // the item's first piece
          p.meta[2 * w.item] = w.first;
          p.meta[2 * w.item + 1] = w.n;
        }
      } else if (p.balanced && threadIdx.x == 64) {
        p.meta[2 * w.item] = (int)blockIdx.x;
        p.meta[2 * w.item + 1] = 1;
      }
#pragma unroll 1
      for (int c0 = 0; c0 < DV; c0 += 32) {
        uint32_t v[32];
        if (ntiles > 0) {
          tmem_ld32(t_lane + C::OCOL + c0, v);  // the whole warp loads; rows past R store nothing
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) v[c] = 0u;  // no key in this block's range: zero rows
        }
        if (!row_ok) continue;
        if (whole) {  // final bf16 rows
          uint4* d4 = reinterpret_cast<uint4*>(p.out + rowflat * DV + c0);
#pragma unroll
          for (int u = 0; u < 4; ++u)
            d4[u] = make_uint4(pack_bf16(__uint_as_float(v[8 * u + 0]) * inv, __uint_as_float(v[8 * u + 1]) * inv),
                               pack_bf16(__uint_as_float(v[8 * u + 2]) * inv, __uint_as_float(v[8 * u + 3]) * inv),
                               pack_bf16(__uint_as_float(v[8 * u + 4]) * inv, __uint_as_float(v[8 * u + 5]) * inv),
                               pack_bf16(__uint_as_float(v[8 * u + 6]) * inv, __uint_as_float(v[8 * u + 7]) * inv));
        } else {  // fp32 partial of this piece, for the combine
          float4* d4 = reinterpret_cast<float4*>(part_o + c0);
#pragma unroll
          for (int u = 0; u < 8; ++u)
            d4[u] = make_float4(__uint_as_float(v[4 * u + 0]) * inv, __uint_as_float(v[4 * u + 1]) * inv,
                                __uint_as_float(v[4 * u + 2]) * inv, __uint_as_float(v[4 * u + 3]) * inv);
        }
      }
      if (row_ok) {
        if (whole) {
          if (p.lse) p.lse[rowflat] = lse_val;
        } else {
          *part_l = lse_val;
        }
      }
    }
  }

  // ---- teardown: nothing of this CTA is in flight
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace

bool gqa_prefill_supported(int dk, int dv, bool fp8) {
  if (fp8) return dk == dv && (dk == 128 || dk == 256);
  return (dv == 128 && (dk == 128 || dk == 192)) || (dk == 256 && dv == 256);
}

template <int DK, int DV, bool FP8>
static cudaError_t launch_pf(const GqaLaunch& a, cudaStream_t stream) {
  using C = PfCfg<DK, DV, FP8>;
  static std::atomic<unsigned long long> smem_limit_set{0};
  if (cudaError_t e = ensure_smem_limit(gqa_prefill_kernel<DK, DV, FP8>, C::SMEM, smem_limit_set)) return e;
  CUtensorMap tq, tk, tv;
  {  // queries as [b*Hq*s rows, DK]: boxes [128 rows x 64 values]
    const cuuint64_t dims[2] = {(cuuint64_t)DK, (cuuint64_t)a.b * a.hq * a.s};
    const cuuint64_t strides[1] = {(cuuint64_t)DK * 2};
    const cuuint32_t box[2] = {64, PM};
    if (!encode_tmap_bf16_sw128(&tq, a.q, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  const uint64_t tokens = a.paged ? (uint64_t)a.num_pages * PK : (uint64_t)a.b * a.capacity;
  if constexpr (FP8) {
    // E4M3 K and V [tokens, KV heads, width] bytes: a box {width, 1 head, 64 tokens} lands
    // as [64 rows][width bytes], unswizzled (the widening warps read it row by row)
    const cuuint32_t kbox[3] = {(cuuint32_t)DK, 1, PK};
    const cuuint32_t vbox[3] = {(cuuint32_t)DV, 1, PK};
    const cuuint64_t kdims[3] = {(cuuint64_t)DK, (cuuint64_t)a.hkv, (cuuint64_t)tokens};
    const cuuint64_t kstrides[2] = {(cuuint64_t)DK, (cuuint64_t)a.hkv * DK};
    const cuuint64_t vdims[3] = {(cuuint64_t)DV, (cuuint64_t)a.hkv, (cuuint64_t)tokens};
    const cuuint64_t vstrides[2] = {(cuuint64_t)DV, (cuuint64_t)a.hkv * DV};
    if (!encode_tmap_u8(&tk, a.k, 3, kdims, kstrides, kbox) || !encode_tmap_u8(&tv, a.v, 3, vdims, vstrides, vbox))
      return cudaErrorInvalidValue;
  } else {
    // K and V [tokens, KV heads, width] viewed as {64 values, tokens, width / 64 chunks, KV
    // heads} (strides: token hkv*width*2 B, chunk 128 B, head width*2 B): a box {64, 64
    // tokens, all chunks, 1 head} lands chunk-major, each 128-byte row swizzled
    const cuuint32_t kbox[4] = {64, PK, (cuuint32_t)C::KCH, 1};
    const cuuint32_t vbox[4] = {64, PK, (cuuint32_t)C::VCH, 1};
    const cuuint64_t kdims[4] = {64, (cuuint64_t)tokens, (cuuint64_t)C::KCH, (cuuint64_t)a.hkv};
    const cuuint64_t kstrides[3] = {(cuuint64_t)a.hkv * DK * 2, 128, (cuuint64_t)DK * 2};
    const cuuint64_t vdims[4] = {64, (cuuint64_t)tokens, (cuuint64_t)C::VCH, (cuuint64_t)a.hkv};
    const cuuint64_t vstrides[3] = {(cuuint64_t)a.hkv * DV * 2, 128, (cuuint64_t)DV * 2};
    if (!encode_tmap_bf16_sw128(&tk, a.k, 4, kdims, kstrides, kbox) ||
        !encode_tmap_bf16_sw128(&tv, a.v, 4, vdims, vstrides, vbox))
      return cudaErrorInvalidValue;
  }
  PfParams p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.lse = a.lse;
  p.seqlens = a.seqlens;
  p.block_table = a.block_table;
  p.max_pages = a.max_pages;
  p.paged = a.paged;
  p.capacity = a.capacity;
  p.num_pages = a.num_pages;
  p.b = a.b;
  p.s = a.s;
  p.hq = a.hq;
  p.hkv = a.hkv;
  p.G = a.hq / a.hkv;
  p.R = p.G * a.s;
  p.nrb = (p.R + PM - 1) / PM;
  p.nsplit = a.nsplit;
  p.chunk = a.chunk;
  p.ws_o = a.ws_o;
  p.ws_lse = a.ws_lse;
  p.balanced = a.balanced_grid > 0 ? 1 : 0;
  p.meta = a.meta;
  p.scale_log2 = a.scale * (FP8 ? a.k_scale : 1.f) * kPLog2e;
  p.v_scale = FP8 ? a.v_scale : 1.f;
  p.err = a.err;
  p.wait_ns = a.wait_ns;
  p.test_timeout = a.test_timeout;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = p.balanced ? dim3(a.balanced_grid) : dim3(p.nrb * p.nsplit, a.hkv, a.b);
  cfg.blockDim = dim3(pf_threads(FP8));
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, gqa_prefill_kernel<DK, DV, FP8>, tq, tk, tv, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_gqa_prefill(const GqaLaunch& a, cudaStream_t stream) {
  if (a.fp8) {
    if (a.dk == 128 && a.dv == 128) return launch_pf<128, 128, true>(a, stream);
    if (a.dk == 256 && a.dv == 256) return launch_pf<256, 256, true>(a, stream);
    return cudaErrorInvalidValue;
  }
  if (a.dk == 192 && a.dv == 128) return launch_pf<192, 128, false>(a, stream);
  if (a.dk == 128 && a.dv == 128) return launch_pf<128, 128, false>(a, stream);
  if (a.dk == 256 && a.dv == 256) return launch_pf<256, 256, false>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace decattn
