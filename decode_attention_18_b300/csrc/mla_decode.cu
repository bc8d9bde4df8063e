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
//       - the S CTA (cluster rank 0) keeps Q' = [Qz | q_pe] of its 128 rows in
//         Tensor Memory (288 columns) as the A operand and computes
//         S = Q' K'^T one 64-key tile (one page) at a time into three 64-column
//         S buffers (tcgen05.mma kind::f16, M=128 N=64, B = the K' chunks in
//         shared memory); four softmax warps (thread = row) turn S into P (bf16)
//         and ship it, with the row rescale factors, to the O CTA's shared memory
//         in one bulk copy per tile (cp.async.bulk shared::cta -> shared::cluster,
//         completing on the O CTA's mbarrier);
//       - the O CTA (rank 1) keeps the whole fp32 O_lat [128 x 512] in Tensor
//         Memory and accumulates O += P Z (M=128 N=256 K=16, A = P and B = the
//         Z slab, both in shared memory), streaming Z itself; its MMA commits
//         free the P buffers of the S CTA (a commit multicast to its mbarrier).
//     Every cache byte enters each SM's shared memory once per tile, and the
//     scores are computed once ("Cost Models", FlashMLA FLOP count).
//   * Cache tiles are 64 keys, one page of a paged pool: TMA boxes of
//     [64 keys x 64 dims] (128-byte swizzle) feed an S-ring (3 chunks per item)
//     and an O-ring ([64 keys x 256 columns] per item).
//   * Online softmax with a lazily moved reference maximum: a row's reference
//     moves only when its maximum grows past it by 2^8 (P stays below 256); the
//     O CTA then rescales those rows of O in Tensor Memory before the tile's
//     MMAs (rare after the first tile). Exponentials use ex2.approx.
//   * Keys past a row's causal limit (token i of s sees keys 0 .. L - s + i)
//     are masked in the softmax; Z rows past the sequence end are zeroed in
//     shared memory before the O MMAs (a cache may hold anything there).
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

#include "common.cuh"
#include "internal.h"

namespace decattn {

namespace {

constexpr int TK = 64;                     // keys per tile (one 64-token page)
constexpr int BM = 128;                    // query rows per row tile (MMA M)
constexpr int NSB = 3;                     // S buffers in Tensor Memory (S CTA)
constexpr int NMSG = 2;                    // P message buffers (staging in S, landing in O)
constexpr int NSMW = 4;                    // softmax warps (S) / rescale + epilogue warps (O)
constexpr int NTHREADS = 32 * (2 + NSMW);  // producer, MMA issuer, NSMW row warps
constexpr int CHUNK = TK * 128;            // one [64 keys x 64 dims] box, 128-byte rows
constexpr int P_TILE = BM * TK * 2;        // P [128 rows x 64 keys] bf16, K-major, 128-byte swizzle
constexpr int MSG_ALPHA = P_TILE;          // [128] float row rescale factors
constexpr int MSG_FLAGS = MSG_ALPHA + BM * 4;  // [NSMW] per-warp "a row was rescaled" words
constexpr int MSG_BYTES = MSG_FLAGS + 16;
constexpr int MSG_STRIDE = 17 * 1024;      // 1024-byte aligned message slots
constexpr int FIN_BYTES = BM * 4;          // [128] float 1/l, sent once at the end
constexpr int S_NR = 7;                    // S-ring slots
constexpr int O_NR = 5;                    // O-ring slots
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.f;                        // move the reference max only past 2^8
constexpr unsigned long long kTeardownNs = 1000000000ull;  // 1 s for own copies / MMAs at exit
constexpr unsigned long long kTestWaitNs = 1000000ull;     // 1 ms forced-timeout wait
constexpr uint32_t kRankS = 0, kRankO = 1;
constexpr int kBarA = 1, kBarB = 2;        // named barriers of the softmax warps

static_assert(MSG_BYTES % 16 == 0 && MSG_BYTES <= MSG_STRIDE, "message");

constexpr int cmax(int a, int b) { return a > b ? a : b; }

template <int KL, int P>
struct MlaCfg {
  static constexpr int NBL = KL / 64;                   // latent chunks per tile
  static constexpr int NCH = NBL + 1;                   // + the RoPE chunk
  static constexpr int CPI = NCH % 3 == 0 ? 3 : NCH;    // chunks per S-ring item
  static constexpr int NITEM = NCH / CPI;               // S-ring items per tile
  static constexpr int S_ITEM = CPI * CHUNK;
  static constexpr int PE_ROW = P * 2;                  // bytes per RoPE row
  static constexpr uint32_t PE_SWZ = PE_ROW == 128 ? kSw128 : (PE_ROW == 64 ? kSw64 : kSw32);
  static constexpr int PE_BOX = TK * PE_ROW;
  static constexpr int ON = KL < 256 ? KL : 256;        // O MMA N (columns per O-ring item)
  static constexpr int NH = KL / ON;                    // O column blocks
  static constexpr int O_ITEM = TK * ON * 2;            // [64 keys x ON columns]
  static constexpr int QC = (KL + P) / 2;               // Tensor Memory columns of Q'
  static constexpr int SB0 = (QC + 31) & ~31;           // first S buffer column
  static constexpr int OFF_MSG = 0;                     // same offset in both CTAs (peer-addressed)
  static constexpr int OFF_RING = NMSG * MSG_STRIDE;
  static constexpr int RING_END = cmax(OFF_RING + S_NR * S_ITEM, OFF_RING + O_NR * O_ITEM);
  static constexpr int OFF_FIN = RING_END;              // same offset in both CTAs
  static constexpr int OFF_BAR = OFF_FIN + FIN_BYTES;   // same offset in both CTAs
  static constexpr int SMEM = OFF_BAR + 512;
  static_assert(KL % 64 == 0 && KL % ON == 0 && ON % 16 == 0 && ON <= 256, "latent width");
  static_assert(P % 16 == 0 && PE_ROW <= 128, "rope width");
  static_assert(NCH % CPI == 0 && CPI <= 32, "S-ring items");
  static_assert(SB0 + NSB * TK <= 512 && KL <= 512, "tensor memory");
  static_assert(S_ITEM % 1024 == 0 && O_ITEM % 1024 == 0 && OFF_RING % 1024 == 0, "swizzle alignment");
  static_assert(4 * 32 * 512 <= O_NR * O_ITEM || KL < 128, "epilogue staging");
  static_assert(SMEM <= 232448, "shared memory");
};

// barrier slots (8 bytes each) at OFF_BAR, the same in both CTAs
enum : int {
  B_FULL = 0,       // [S_NR] ring item landed
  B_EMPTY = 7,      // [S_NR] ring item consumed
  B_SFULL = 14,     // [NSB] S tile in Tensor Memory (S CTA)
  B_SEMPTY = 17,    // [NSB] S tile read by the softmax warps (S CTA)
  B_PFULL = 20,     // [NMSG] P message landed (O CTA; the S CTA's copy completes on it)
  B_PFREE = 22,     // [NMSG] O CTA's MMAs done with message buffer (S CTA; O's commit arrives)
  B_QREADY = 24,    // Q' in Tensor Memory (S CTA)
  B_FINFULL = 25,   // 1/l landed (O CTA)
  B_ODONE = 26,     // every O MMA issued before a rescale complete (O CTA)
  B_OFINAL = 27,    // every O MMA complete (O CTA)
  B_CREQ = 28,      // rescale request (or end marker) for the row warps (O CTA)
  B_CDONE = 29,     // rescale done (O CTA)
  B_TEST = 30,      // never signalled: the forced-timeout test waits on it
  B_FIN = 31,       // teardown: every tcgen05 op of the MMA issuer complete
  B_COUNT = 32
};
static_assert(S_NR <= 7 && O_NR <= 7, "ring barrier slots");

struct MlaParams {
  const __nv_bfloat16* qz;
  const __nv_bfloat16* q_pe;
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

// cache row of `key` of sequence bi (paged: through the block table; a tile never
// crosses a page because tiles and pages are both 64 keys and chunks are whole tiles)
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

template <int KL, int P>
__global__ void __launch_bounds__(NTHREADS, 1)
    mla_pair_kernel(const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_kpe,
                    MlaParams p) {
  using C = MlaCfg<KL, P>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sb = smem_u32(smem);
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = blockIdx.x >> 1;  // row tile (one cluster each)
  const int split = blockIdx.y;
  const int bi = blockIdx.z;
  const int kstart = split * p.chunk;
  const int qrow0 = bi * p.rows + mt * BM;  // first flattened [b*h*s] query row of the tile

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + B_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + B_COUNT) + 1;
  volatile int* req_tile = reinterpret_cast<volatile int*>(bars + B_COUNT) + 2;
  auto msg = [&](int m) { return smem + C::OFF_MSG + m * MSG_STRIDE; };

  // ---- set-up that touches no global memory (overlaps the previous kernel's end)
  if (threadIdx.x == 0) {
    for (int i = 0; i < 7; ++i) {
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
    mbar_init(&bars[B_QREADY], NSMW);
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
    prefetch_tmap(&tm_z);
    prefetch_tmap(&tm_kpe);
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
  if (kstart >= L && L <= 0 && p.nsplit == 1) {  // empty sequence without a combine pass
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
  const int kend = min(L, kstart + p.chunk);
  const int ntiles = active ? (kend - kstart + TK - 1) / TK : 0;
  constexpr uint32_t tmem = 0;

  if (rank == kRankS) {
    // =====================================================================================
    // S CTA
    if (warp == 0) {
      // ------------------------------------------------ producer: K' chunks into the S-ring
      // The whole warp walks the items (warp-uniform values); lane 0 arms the item's
      // barrier and lanes 0..CPI-1 each request one chunk box.
      RingPos<S_NR> rp;
      int ic = 0;
      int last[S_NR];
      for (int i = 0; i < S_NR; ++i) last[i] = -1;
      bool ok = true;
      for (int t = 0; ok && t < ntiles; ++t) {
        const int row0 = cache_row(p, bi, kstart + t * TK);
        for (int it = 0; it < C::NITEM; ++it) {
          const int slot = rp.slot;
          const uint32_t prev = rp.phase ^ 1u;
          rp.advance();
          if (ic >= S_NR && !warp_wait(&bars[B_EMPTY + slot], prev, p.wait_ns, abort_flag)) {
            ok = false;
            break;
          }
          last[slot] = ic++;
          const bool has_pe = it == C::NITEM - 1;
          const uint32_t bytes = has_pe ? (C::CPI - 1) * CHUNK + C::PE_BOX : C::CPI * CHUNK;
          if (lane == 0) mbar_expect_tx(&bars[B_FULL + slot], bytes);
          __syncwarp();
          if (lane < C::CPI) {
            const int j = it * C::CPI + lane;
            const uint32_t dst = sb + C::OFF_RING + slot * C::S_ITEM + lane * CHUNK;
            if (j < C::NBL)
              tma_load_2d(dst, &tm_z, j * 64, row0, &bars[B_FULL + slot]);
            else
              tma_load_2d(dst, &tm_kpe, 0, row0, &bars[B_FULL + slot]);
          }
          __syncwarp();
        }
      }
      if (lane == 0) {
        if (!ok && !*abort_flag) fail();
        for (int i = 0; i < S_NR; ++i)  // no copy may still be landing when the CTA exits
          if (last[i] >= 0) mbar_wait(&bars[B_FULL + i], (last[i] / S_NR) & 1, kTeardownNs, nullptr);
      }
      __syncwarp();
    } else if (warp == 1) {
      // ------------------------------------------------ MMA issuer: S = Q' K'^T
      bool ok = ntiles == 0 || warp_wait(&bars[B_QREADY], 0, p.wait_ns, abort_flag);
      if (ok && ntiles > 0 && p.test_timeout) ok = warp_wait(&bars[B_TEST], 0, kTestWaitNs, abort_flag);
      tc_fence_after();  // Q' was written to Tensor Memory by the softmax warps
      const bool leader = elect_one();
      constexpr uint32_t idS = idesc_bf16_f32(BM, TK, false, false);
      const uint64_t dring = smem_desc(sb + C::OFF_RING, 16, 1024, kSw128);
      const uint64_t dring_pe = smem_desc(sb + C::OFF_RING, 16, 8 * C::PE_ROW, C::PE_SWZ);
      RingPos<S_NR> rp;
      for (int t = 0; ok && t < ntiles; ++t) {
        const int buf = t % NSB;
        if (t >= NSB && !warp_wait(&bars[B_SEMPTY + buf], ((t / NSB) - 1) & 1, p.wait_ns, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();  // the softmax warps' loads of this buffer come first
        const uint32_t d_s = tmem + C::SB0 + buf * TK;
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
            for (int c = 0; c < C::CPI; ++c) {
              const int j = it * C::CPI + c;
              const uint64_t so = (uint64_t)((slot * C::S_ITEM + c * CHUNK) >> 4);
              if (j < C::NBL) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  tc_mma_ts(d_s, tmem + j * 32 + kk * 8, dring + so + 2 * kk, idS, (j | kk) ? 1u : 0u);
              } else {
#pragma unroll
                for (int kk = 0; kk < P / 16; ++kk)
                  tc_mma_ts(d_s, tmem + KL / 2 + kk * 8, dring_pe + so + 2 * kk, idS, 1u);
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
      // ------------------------------------------------ Q' load, softmax, P messages (warps 2-5)
      const int q = warp & 3;  // Tensor Memory lane quadrant this warp may access
      const int r = q * 32 + lane;
      const int row_in_seq = mt * BM + r;
      const bool row_ok = row_in_seq < p.rows;
      const int lim = row_ok ? min(kend, L - p.s + (row_in_seq % p.s) + 1) : 0;  // exclusive key limit
      const uint32_t t_lane = tmem + ((uint32_t)(q * 32) << 16);
      const size_t grow = (size_t)qrow0 + r;
      const bool issuer = warp == 2 && lane == 0;
      if (ntiles > 0) {
        // Q' row r into Tensor Memory (A operand: lane = row, two bf16 per column, even k low)
#pragma unroll 1
        for (int c0 = 0; c0 < C::NBL; ++c0) {
          uint32_t v[32];
          const uint4* src = reinterpret_cast<const uint4*>(p.qz + grow * KL + c0 * 64);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const uint4 x = row_ok ? __ldg(src + e) : make_uint4(0, 0, 0, 0);
            v[4 * e] = x.x;
            v[4 * e + 1] = x.y;
            v[4 * e + 2] = x.z;
            v[4 * e + 3] = x.w;
          }
          tmem_st32(t_lane + c0 * 32, v);
        }
        {
          const uint4* src = reinterpret_cast<const uint4*>(p.q_pe + grow * P);
          uint32_t v[32];
#pragma unroll
          for (int e = 0; e < P / 8; ++e) {
            const uint4 x = row_ok ? __ldg(src + e) : make_uint4(0, 0, 0, 0);
            v[4 * e] = x.x;
            v[4 * e + 1] = x.y;
            v[4 * e + 2] = x.z;
            v[4 * e + 3] = x.w;
          }
          if constexpr (P == 64)
            tmem_st32(t_lane + KL / 2, v);
          else
            tmem_st8(t_lane + KL / 2, v);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[B_QREADY]);
      }
      const uint32_t peer_msg0 = mapa_shared(sb + C::OFF_MSG, peer);
      const uint32_t peer_pfull0 = mapa_shared(smem_u32(&bars[B_PFULL]), peer);
      float m_ref = -INFINITY, l_run = 0.f;
      bool ok = true;
      for (int t = 0; t < ntiles; ++t) {
        const int buf = t % NSB;
        const int m = t % NMSG;
        const bool okw = warp_wait(&bars[B_SFULL + buf], (t / NSB) & 1, p.wait_ns, abort_flag);
        float x[TK];
        float alpha = 1.f;
        uint32_t pk[TK / 2];
        if (okw) {
          tc_fence_after();
          uint32_t sv[32];
          const uint32_t sbuf = t_lane + C::SB0 + buf * TK;
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
          const int kb = kstart + t * TK;
          if (kb + TK > lim) {
#pragma unroll
            for (int c = 0; c < TK; ++c)
              if (kb + c >= lim) x[c] = -INFINITY;
          }
          float m8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) m8[e] = x[e];
#pragma unroll
          for (int c = 8; c < TK; ++c) m8[c & 7] = fmaxf(m8[c & 7], x[c]);
          const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                 fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
          if (mx > m_ref + kRescaleLog2) {
            alpha = fast_exp2(m_ref - mx);  // 0 when nothing was seen yet
            m_ref = mx;
            l_run *= alpha;
          }
          const float mneg = m_ref == -INFINITY ? 0.f : -m_ref;  // all keys masked so far: x = -inf -> 0
          float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int e = 0; e < TK / 2; ++e) {
            const float p0 = fast_exp2(x[2 * e] + mneg);
            const float p1 = fast_exp2(x[2 * e + 1] + mneg);
            ps[e & 3] += p0 + p1;
            pk[e] = pack_bf16(p0, p1);
          }
          l_run += (ps[0] + ps[1]) + (ps[2] + ps[3]);
        }
        // every softmax warp arrives here on every tile, whatever its wait did, so that
        // all leave the loop together; the issuer has released staging slot m (below)
        if (!named_bar_and(kBarA, 32 * NSMW, okw && !*abort_flag)) {
          ok = false;
          break;
        }
        // P row r into staging slot m: 128-byte row, 16-byte unit u at (u ^ (r & 7))
        uint8_t* st = msg(m);
#pragma unroll
        for (int u = 0; u < 8; ++u)
          *reinterpret_cast<uint4*>(st + r * 128 + ((u ^ (r & 7)) << 4)) =
              make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        // the first tile fills an empty O (its MMAs do not accumulate): nothing to rescale
        const float a_out = t == 0 ? 1.f : alpha;
        reinterpret_cast<float*>(st + MSG_ALPHA)[r] = a_out;
        const bool any = __any_sync(0xffffffffu, a_out != 1.f);
        if (lane == 0) reinterpret_cast<int*>(st + MSG_FLAGS)[warp - 2] = any ? 1 : 0;
        fence_proxy_async_smem();  // the bulk copy (async proxy) reads what these stores wrote
        named_bar_sync(kBarB, 32 * NSMW);
        if (issuer) {
          // the O CTA's MMAs are done with its message buffer m (tile t - NMSG)
          const bool free_ok =
              t < NMSG || mbar_wait(&bars[B_PFREE + m], ((t / NMSG) - 1) & 1, p.wait_ns, abort_flag);
          if (free_ok) {
            bulk_copy_to_peer(peer_msg0 + m * MSG_STRIDE, sb + C::OFF_MSG + m * MSG_STRIDE, MSG_BYTES,
                              peer_pfull0 + m * 8);
            bulk_commit();
            bulk_wait_read<NMSG - 1>();  // staging slot (t + 1) % NMSG is free for the next tile
          } else if (!*abort_flag) {
            fail();
          }
        }
      }
      ok = named_bar_and(kBarA, 32 * NSMW, ok && !*abort_flag);
      const float lse = l_run > 0.f ? (m_ref + log2f(l_run)) * kLn2 : -INFINITY;
      if (ok && ntiles > 0) {
        if (row_ok) {
          if (p.nsplit == 1) {
            if (p.lse) p.lse[grow] = lse;
          } else {
            p.ws_lse[grow * p.nsplit + split] = lse;
          }
        }
        reinterpret_cast<float*>(smem + C::OFF_FIN)[r] = l_run > 0.f ? 1.f / l_run : 0.f;
        fence_proxy_async_smem();
      }
      named_bar_sync(kBarB, 32 * NSMW);
      if (issuer) {
        if (ok && ntiles > 0) {
          bulk_copy_to_peer(mapa_shared(sb + C::OFF_FIN, peer), sb + C::OFF_FIN, FIN_BYTES,
                            mapa_shared(smem_u32(&bars[B_FINFULL]), peer));
          bulk_commit();
        }
        bulk_wait<0>();  // every copy into the peer has landed
        // the O CTA's last commits into this CTA's barriers have arrived
        if (ok)
          for (int t = ntiles > NMSG ? ntiles - NMSG : 0; t < ntiles; ++t)
            if (!mbar_wait(&bars[B_PFREE + t % NMSG], (t / NMSG) & 1, p.wait_ns, abort_flag)) {
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
        const int row0 = cache_row(p, bi, kstart + t * TK);
        for (int nh = 0; nh < C::NH; ++nh) {
          const int slot = rp.slot;
          const uint32_t prev = rp.phase ^ 1u;
          rp.advance();
          if (ic >= O_NR && !warp_wait(&bars[B_EMPTY + slot], prev, p.wait_ns, abort_flag)) {
            ok = false;
            break;
          }
          last[slot] = ic++;
          if (lane == 0) mbar_expect_tx(&bars[B_FULL + slot], C::O_ITEM);
          __syncwarp();
          if (lane < C::ON / 64)
            tma_load_2d(sb + C::OFF_RING + slot * C::O_ITEM + lane * CHUNK, &tm_z, nh * C::ON + lane * 64, row0,
                        &bars[B_FULL + slot]);
          __syncwarp();
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
      const uint64_t dmsg = smem_desc(sb + C::OFF_MSG, 16, 1024, kSw128);      // P, K-major
      const uint64_t dz = smem_desc(sb + C::OFF_RING, CHUNK, 1024, kSw128);    // Z slab, MN-major
      RingPos<O_NR> rp;
      int ncorr = 0;
      bool ok = true;
      for (int t = 0; ok && t < ntiles; ++t) {
        const int m = t % NMSG;
        if (leader) mbar_expect_tx(&bars[B_PFULL + m], MSG_BYTES);  // this use's one arrival + bytes
        __syncwarp();
        if (!warp_wait(&bars[B_PFULL + m], (t / NMSG) & 1, p.wait_ns, abort_flag)) {
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
        for (int nh = 0; nh < C::NH; ++nh) {
          const int slot = rp.slot;
          const uint32_t ph = rp.phase;
          rp.advance();
          if (!warp_wait(&bars[B_FULL + slot], ph, p.wait_ns, abort_flag)) {
            ok = false;
            break;
          }
          const int first_bad = L - key0;  // rows at or past the sequence end may hold anything
          if (first_bad < TK) {
            uint8_t* item = smem + C::OFF_RING + slot * C::O_ITEM;
            const int nrow = TK - first_bad;
            for (int idx = lane; idx < nrow * (C::ON / 64) * 8; idx += 32) {
              const int rr = first_bad + idx / ((C::ON / 64) * 8);
              const int rem = idx % ((C::ON / 64) * 8);
              *reinterpret_cast<uint4*>(item + (rem / 8) * CHUNK + rr * 128 + (rem % 8) * 16) =
                  make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            __syncwarp();
          }
          if (leader) {
            const uint64_t a0 = dmsg + (uint64_t)((m * MSG_STRIDE) >> 4);
            const uint64_t b0 = dz + (uint64_t)((slot * C::O_ITEM) >> 4);
#pragma unroll
            for (int kk = 0; kk < TK / 16; ++kk)
              tc_mma_ss(tmem + nh * C::ON, a0 + 2 * kk, b0 + (uint64_t)((kk * 16 * 128) >> 4), idO,
                        (t > 0 || kk > 0) ? 1u : 0u);
            tc_commit(&bars[B_EMPTY + slot]);
          }
          __syncwarp();
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
      const int r = q * 32 + lane;
      const uint32_t t_lane = tmem + ((uint32_t)(q * 32) << 16);
      bool ok = true;
      for (int k = 0;; ++k) {
        if (!warp_wait(&bars[B_CREQ], k & 1, p.wait_ns, abort_flag)) {
          ok = false;
          break;
        }
        const int tile = *req_tile;
        if (tile < 0) break;
        const float alpha = reinterpret_cast<const volatile float*>(msg(tile % NMSG) + MSG_ALPHA)[r];
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
          tc_fence_after();
#pragma unroll 1
          for (int c0 = 0; c0 < KL; c0 += 32) {
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
          // O / l of this warp's 32 rows is staged through shared memory (the O-ring, idle
          // once every MMA has completed) in passes of 128 columns and stored as whole row
          // segments; staged rows are 16-byte units XOR-swizzled by (row & 7).
          constexpr int PASS = KL < 128 ? KL : 128;
          constexpr int F4 = PASS / 4;  // 16-byte units per staged row
          constexpr int ROWB = PASS * 4;
          constexpr int RPI = 32 / F4;  // rows per store instruction
          uint8_t* stg = smem + C::OFF_RING + (warp - 2) * 32 * ROWB;
#pragma unroll 1
          for (int c0 = 0; c0 < KL; c0 += PASS) {
#pragma unroll 1
            for (int cc = 0; cc < PASS; cc += 32) {
              uint32_t v[32];
              tmem_ld32(t_lane + c0 + cc, v);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 8; ++e)
                *reinterpret_cast<float4*>(stg + lane * ROWB + (((cc / 4 + e) ^ (lane & 7)) * 16)) =
                    make_float4(__uint_as_float(v[4 * e + 0]) * inv, __uint_as_float(v[4 * e + 1]) * inv,
                                __uint_as_float(v[4 * e + 2]) * inv, __uint_as_float(v[4 * e + 3]) * inv);
            }
            __syncwarp();
            const int jl = lane % F4;
#pragma unroll 4
            for (int rr = lane / F4; rr < 32; rr += RPI) {
              const int rs = q * 32 + rr;  // row within the tile
              if (mt * BM + rs >= p.rows) continue;
              const float4 xv = *reinterpret_cast<const float4*>(stg + rr * ROWB + ((jl ^ (rr & 7)) * 16));
              const size_t g = (size_t)qrow0 + rs;
              const int col = c0 + jl * 4;
              if (p.nsplit == 1)
                *reinterpret_cast<uint2*>(p.o_lat + g * KL + col) =
                    make_uint2(pack_bf16(xv.x, xv.y), pack_bf16(xv.z, xv.w));
              else
                *reinterpret_cast<float4*>(p.ws_o + (g * p.nsplit + split) * KL + col) = xv;
            }
            __syncwarp();
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

template <int KL, int P>
cudaError_t launch_kl(const MlaLaunch& a, cudaStream_t stream) {
  using C = MlaCfg<KL, P>;
  static std::atomic<unsigned long long> smem_limit_set{0};
  if (cudaError_t e = ensure_smem_limit(mla_pair_kernel<KL, P>, C::SMEM, smem_limit_set)) return e;
  const uint64_t krows = a.paged ? (uint64_t)a.num_pages * 64 : (uint64_t)a.b * a.capacity;
  CUtensorMap tz, tkpe;
  if (!make_map(&tz, a.z, krows, KL, TK, 64) || !make_map(&tkpe, a.k_pe, krows, P, TK, P))
    return cudaErrorInvalidValue;
  MlaParams p;
  p.qz = static_cast<const __nv_bfloat16*>(a.qz);
  p.q_pe = static_cast<const __nv_bfloat16*>(a.q_pe);
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
  const int mtiles = (p.rows + BM - 1) / BM;
  // a cluster of two CTAs per row tile, launched as a programmatic dependent
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * mtiles, a.nsplit, a.b);
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
  const cudaError_t e = cudaLaunchKernelEx(&cfg, mla_pair_kernel<KL, P>, tz, tkpe, p);
  return e != cudaSuccess ? e : cudaGetLastError();
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
