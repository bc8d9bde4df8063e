// Grouped-head split-KV decode on 5th-generation tensor cores, for KV heads shared by many
// query rows (MQA and wide GQA: G*s between 17 and 32 per row block).
//
// Same computation as gqa.cu ("Why MLA and MTP Fight Each Other", summary table: MHA /
// GQA / MQA are one attention with different KV-head counts; "MHA vs GQA" Q&A section 1:
// a KV head serves Hq/Hkv query heads), laid out for tcgen05 with the KEYS in the MMA M
// dimension, so that the few query rows of a KV head only pad to N = 32:
//   S^T = K Q^T     M = 64 keys, N = 32 rows, K = d            (both operands in smem)
//   O^T += V^T P^T  M = 128 value dims per tile, N = 32 rows, K = 16 keys per step
//                   (V read MN-major from the same shared-memory tile that was loaded
//                   for it, P^T written by the softmax warps into shared memory)
// With each K/V byte feeding 2*32*2 FLOPs through the tensor pipe, the kernel stays bound
// by the cache read even for MQA (24 query rows per KV head).
//
//  * One CTA per (sequence, KV head, context chunk, 32-row block). K and V tiles of 64
//    keys (one 64-token page) stream through a 3-stage ring, loaded by TMA through a 3-D
//    tensor map (d, head, token) in [64 tokens x 64 dims] boxes (128-byte swizzle); two
//    producer warps (K and V) issue them, one thread's bulk copies being served one after
//    another.
//  * Warp 2 issues the MMAs (lane 0) and owns the Tensor Memory (S^T double buffer +
//    O^T accumulator, 128 columns); warps 3-6 run the softmax with thread = key: TMEM
//    lanes 0-15 of each quadrant hold the 64 keys of an M = 64 tile.
//  * Softmax: every row keeps a reference maximum in shared memory that moves only when
//    a key's score exceeds it by more than 2^8 (then O^T columns and partial sums are
//    rescaled); P^T (bf16) goes to a double-buffered shared-memory tile; each thread keeps
//    its partial row sums, reduced once at the end.
//  * Keys past the chunk end are masked; value rows past the sequence end are zeroed in
//    shared memory before the O^T MMA (cache rows past the end may hold anything).
//  * Every mbarrier wait is bounded; on time-out the CTA records the error, winds down
//    (own copies and MMAs), frees Tensor Memory and returns.
// Output: with a single chunk, bf16 rows and LSE directly; otherwise fp32 (O, LSE)
// partials for the combine kernel.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"

namespace decattn {

namespace {

constexpr int TKY = 64;          // keys per tile (M of S^T; one 64-token page)
constexpr int NROW = 32;         // query rows per CTA (N)
constexpr int NST = 3;           // K/V ring stages
constexpr int NPROD = 2;           // producer warps: 0 K (and Q), 1 V
constexpr int MMAW = NPROD;        // MMA-issuing warp
constexpr int SMW0 = NPROD + 1;    // first of the four softmax warps
constexpr int NTHREADS = (NPROD + 5) * 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.f;
constexpr unsigned long long kTeardownNs = 1000000000ull;

struct TcParams {
  const int32_t* seqlens;
  const int32_t* block_table;
  int max_pages, paged, capacity, num_pages;
  int b, s, hq, hkv, G, R, nrb, nsplit, chunk;
  float scale_log2;
  __nv_bfloat16* out;
  float* lse;
  float* ws_o;
  float* ws_lse;
  unsigned* err;
  unsigned long long wait_ns;
};

template <int D>
struct TcCfg {
  static constexpr int NCB = D / 64;                   // 64-dim boxes per row
  static constexpr int BOX = TKY * 128;                // [64 tokens x 64 dims]
  static constexpr int TILE = NCB * BOX;               // one K (or V) tile
  static constexpr int QBOX = NROW * 128;              // [32 rows x 64 dims]
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = NCB * QBOX;             // stages of K tiles
  static constexpr int OFF_V = OFF_K + NST * TILE;     // stages of V tiles
  static constexpr int OFF_P = OFF_V + NST * TILE;     // two P^T tiles [64 keys x 128 B]
  static constexpr int OFF_RED = OFF_P + 2 * TKY * 128;  // m_ref[32] | tile max [4][32] | sums [4][32] | flags
  static constexpr int OFF_BAR = OFF_RED + (NROW + 8 * NROW + 64) * 4;
  static constexpr int SMEM = OFF_BAR + 256;
  static constexpr int NMT = D / 128;                  // O^T M-tiles
  static constexpr int TM_S = 0;                       // S^T buffers: 2 x NROW columns
  static constexpr int TM_O = 2 * NROW;                // O^T: NMT x NROW columns
  static constexpr int TM_COLS = 128;
  static_assert(D % 128 == 0 && TM_O + NMT * NROW <= TM_COLS, "tensor memory");
  static_assert(SMEM <= 232448, "shared memory");
};

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns, volatile int* abort_flag) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, limit_ns, abort_flag));
}

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1)
    gqa_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, TcParams p) {
  using C = TcCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sb = smem_u32(smem);
  if (sb & 1023u) {
    if (threadIdx.x == 0) raise_error(p.err, kErrLaunch);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rb = blockIdx.x % p.nrb;
  const int split = blockIdx.x / p.nrb;
  const int g = blockIdx.y;
  const int bi = blockIdx.z;
  const int L = p.seqlens[bi];
  const int kstart = split * p.chunk;
  const int row0 = rb * NROW;                       // first row of the KV head's R rows
  const int nrows = min(NROW, p.R - row0);          // valid rows of this block
  auto out_row = [&](int r) -> size_t {             // flattened [b, Hq, s] index of block row r
    const int rg = row0 + r;
    return (size_t)(bi * p.hq + g * p.G + rg / p.s) * p.s + (rg % p.s);
  };
  if (kstart >= L) {
    if (L <= 0 && p.nsplit == 1) {
      for (int idx = threadIdx.x; idx < nrows * (D / 8); idx += blockDim.x) {
        const int r = idx / (D / 8);
        *reinterpret_cast<uint4*>(p.out + out_row(r) * D + (idx % (D / 8)) * 8) = make_uint4(0, 0, 0, 0);
        if (p.lse && idx % (D / 8) == 0) p.lse[out_row(r)] = -INFINITY;
      }
    }
    return;
  }
  const int kend = min(L, kstart + p.chunk);
  const int ntiles = (kend - kstart + TKY - 1) / TKY;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;   // [NST]
  uint64_t* v_full = bars + 4;   // [NST]
  uint64_t* kv_empty = bars + 7; // [NST] (S^T and O^T of the stage's tile done)
  uint64_t* s_ready = bars + 10; // [2]
  uint64_t* p_full = bars + 12;  // [2] P^T written (+ O^T rescaled)
  uint64_t* p_free = bars + 14;  // [2] O^T of the P^T buffer's tile done
  uint64_t* fin_bar = bars + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 17);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 18);
  float* m_ref = reinterpret_cast<float*>(smem + C::OFF_RED);  // [NROW]
  float* tmax = m_ref + NROW;                                   // [4][NROW]
  float* tsum = tmax + 4 * NROW;                                // [4][NROW]
  volatile int* flags = reinterpret_cast<volatile int*>(tsum + 4 * NROW);  // [0..3] rescale votes, [4..7] ok

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < NST; ++i) {
      mbar_init(&k_full[i], NPROD / 2);
      mbar_init(&v_full[i], NPROD / 2);
      mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_ready[i], 1);
      mbar_init(&p_full[i], 4);
      mbar_init(&p_free[i], 1);
    }
    mbar_init(fin_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (threadIdx.x < NROW) m_ref[threadIdx.x] = -INFINITY;
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  if (warp == MMAW) {
    tmem_alloc(tmem_slot, C::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto fail = [&]() {
    raise_error(p.err, kErrWaitTimeout);
    *abort_flag = 1;
  };
  auto token_row = [&](int key0) -> int {  // cache token row of a tile's first key
    if (p.paged) {
      int page = p.block_table[(size_t)bi * p.max_pages + key0 / TKY];
      if (page < 0 || page >= p.num_pages) {
        raise_error(p.err, kErrBadPage);
        page = 0;
      }
      return page * TKY;
    }
    return bi * p.capacity + key0;
  };

  if (warp < NPROD) {
    // ------------------------------------------------------------ producers: first half K (and Q), second half V
    if (lane == 0) {
      const bool isk = warp < NPROD / 2;
      const int half = warp % (NPROD / 2);  // this warp's share of a tile's boxes
      if (warp == 0) {
        mbar_expect_tx(q_full, C::NCB * C::QBOX);
        const int qrow = (bi * p.hq + g * p.G) * p.s + row0;  // first row of the block in [b*Hq*s, D]
        for (int c = 0; c < C::NCB; ++c) tma_load_2d(sb + C::OFF_Q + c * C::QBOX, &tm_q, c * 64, qrow, q_full);
      }
      uint64_t* full = isk ? k_full : v_full;
      const CUtensorMap* tm = isk ? &tm_k : &tm_v;
      const uint32_t base = sb + (isk ? C::OFF_K : C::OFF_V);
      bool ok = true;
      int last = -1;
      for (int t = 0; ok && t < ntiles; ++t) {
        const int st = t % NST;
        if (t >= NST && !mbar_wait(&kv_empty[st], ((t / NST) - 1) & 1, p.wait_ns, abort_flag)) {
          ok = false;
          break;
        }
        const int trow = token_row(kstart + t * TKY);
        mbar_expect_tx(&full[st], C::TILE / (NPROD / 2));
        for (int c = half; c < C::NCB; c += NPROD / 2) tma_load_3d(base + st * C::TILE + c * C::BOX, tm, c * 64, g, trow, &full[st]);
        last = t;
      }
      if (!ok && !*abort_flag) fail();
      if (warp == 0) mbar_wait(q_full, 0, kTeardownNs, nullptr);
      if (last >= 0) mbar_wait(&full[last % NST], (last / NST) & 1, kTeardownNs, nullptr);
    }
    __syncwarp();
  } else if (warp == MMAW) {
    // ------------------------------------------------------------ MMA issuer (lane 0; the warp zeroes value tails)
    constexpr uint32_t idS = idesc_bf16_f32(TKY, NROW, false, false);
    constexpr uint32_t idO = idesc_bf16_f32(128, NROW, true, true);
    bool ok = warp_wait(q_full, 0, p.wait_ns, abort_flag);
    tc_fence_after();
    const uint64_t dq = smem_desc(sb + C::OFF_Q, 16, 1024, kSw128);
    const uint64_t dk = smem_desc(sb + C::OFF_K, 16, 1024, kSw128);
    const uint64_t dv = smem_desc(sb + C::OFF_V, C::BOX, 1024, kSw128);   // V^T: MN-major, 64-dim groups BOX apart
    const uint64_t dp = smem_desc(sb + C::OFF_P, 16, 1024, kSw128);       // P^T: MN-major, one 128 B group
    auto issue_o = [&](int u) {  // O^T += V_u^T P_u^T (P^T of tile u is complete)
      const int st = u % NST;
      const int first_bad = L - (kstart + u * TKY);  // value rows at or past the sequence end
      if (first_bad < TKY) {
        for (int idx = lane; idx < (TKY - first_bad) * C::NCB * 8; idx += 32) {
          const int rr = first_bad + idx / (C::NCB * 8);
          const int rem = idx % (C::NCB * 8);
          *reinterpret_cast<uint4*>(smem + C::OFF_V + st * C::TILE + (rem / 8) * C::BOX + rr * 128 + (rem % 8) * 16) =
              make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (lane == 0) {
        tc_fence_after();
        const uint64_t vo = (uint64_t)((st * C::TILE) >> 4);
        const uint64_t po = (uint64_t)(((u & 1) * TKY * 128) >> 4);
#pragma unroll
        for (int mi = 0; mi < C::NMT; ++mi)
#pragma unroll
          for (int kk = 0; kk < TKY / 16; ++kk)
            tc_mma_ss(tmem + C::TM_O + mi * NROW, dv + vo + (uint64_t)((mi * 2 * C::BOX + kk * 16 * 128) >> 4),
                      dp + po + (uint64_t)((kk * 16 * 128) >> 4), idO, (u > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&kv_empty[st]);
        tc_commit(&p_free[u & 1]);
      }
      __syncwarp();
    };
    auto issue_s = [&](int t) {  // S^T_t = K_t Q^T (K and V of tile t landed)
      if (lane == 0) {
        tc_fence_after();
        const uint64_t ko = (uint64_t)(((t % NST) * C::TILE) >> 4);
#pragma unroll
        for (int c = 0; c < C::NCB; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_ss(tmem + C::TM_S + (t & 1) * NROW, dk + ko + (uint64_t)((c * C::BOX) >> 4) + 2 * kk,
                      dq + (uint64_t)((c * C::QBOX) >> 4) + 2 * kk, idS, (c > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&s_ready[t & 1]);
      }
      __syncwarp();
    };
    // Issue S^T(t) and O^T(t-1) in whichever order their inputs arrive (O^T frees a ring
    // stage for the producers; S^T feeds the softmax). Lane 0 polls; the warp follows.
    for (int t = 0; ok && t <= ntiles; ++t) {
      bool s_done = t >= ntiles, o_done = t == 0;
      const uint64_t t0 = global_ns();
      while (!(s_done && o_done)) {
        int pick = 0;  // 1: O^T(t-1), 2: S^T(t)
        if (lane == 0) {
          if (!o_done && mbar_test(&p_full[(t - 1) & 1], ((t - 1) >> 1) & 1)) pick = 1;
          else if (!s_done && mbar_test(&k_full[t % NST], (t / NST) & 1) && mbar_test(&v_full[t % NST], (t / NST) & 1))
            pick = 2;
          else if (*abort_flag || global_ns() - t0 > p.wait_ns) pick = 3;
        }
        pick = __shfl_sync(0xffffffffu, pick, 0);
        if (pick == 1) {
          issue_o(t - 1);
          o_done = true;
        } else if (pick == 2) {
          issue_s(t);
          s_done = true;
        } else if (pick == 3) {
          ok = false;
          break;
        }
      }
    }
    if (lane == 0) {
      if (!ok && !*abort_flag) fail();
      tc_commit(fin_bar);
      mbar_wait(fin_bar, 0, kTeardownNs, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax + epilogue (warps 3-6, thread = key)
    const int q = warp & 3;                 // TMEM lane quadrant
    const int sw = warp - SMW0;             // softmax warp index 0..3
    const bool kt = lane < 16;              // lanes 16-31 of an M = 64 tile hold no key
    const int kin = q * 16 + (lane & 15);   // key within the tile (M = 64 layout)
    const uint32_t t_lane = tmem + ((uint32_t)(q * 32) << 16);
    float psum[NROW];
    int lim[NROW];    // exclusive key limit per row (causal among the s new tokens), -1 for padding rows
    float mr8[NROW];  // reference maximum + 2^8 threshold, per row (registers; refreshed after a move)
    float mrz[NROW];  // reference maximum used in the exponent (0 while a row has seen nothing)
#pragma unroll
    for (int r = 0; r < NROW; ++r) {
      psum[r] = 0.f;
      const int rg = row0 + r;
      lim[r] = (r < nrows && kt) ? min(kend, L - p.s + (rg % p.s) + 1) : -1;
      mr8[r] = -INFINITY;
      mrz[r] = 0.f;
    }
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      const bool okw = warp_wait(&s_ready[t & 1], (t >> 1) & 1, p.wait_ns, abort_flag);
      const int key = kstart + t * TKY + kin;
      float x[NROW];
      bool need = false;
      if (okw) {
        tc_fence_after();
        uint32_t sv[32];
        tmem_ld32(t_lane + C::TM_S + (t & 1) * NROW, sv);
        tmem_ld_wait();
#pragma unroll
        for (int r = 0; r < NROW; ++r) {
          const float v = key < lim[r] ? __uint_as_float(sv[r]) * p.scale_log2 : -INFINITY;
          x[r] = v;
          need |= v > mr8[r];
        }
      }
      // one vote per warp, then all four softmax warps agree (named barrier over 128 threads)
      const bool wneed = __any_sync(0xffffffffu, need);
      if (lane == 0) {
        flags[sw] = wneed ? 1 : 0;
        flags[4 + sw] = okw ? 1 : 0;
      }
      named_bar_sync(1, 128);
      const bool any_need = flags[0] | flags[1] | flags[2] | flags[3];
      const bool all_ok = flags[4] & flags[5] & flags[6] & flags[7];
      if (!all_ok) {
        ok = false;
        break;
      }
      if (any_need) {
        // rare: new row maxima over the tile; rescale O^T columns and partial sums. Every
        // barrier below is reached by all four warps; a failed wait only clears `okr`.
        bool okr = true;
#pragma unroll
        for (int r = 0; r < NROW; ++r) {
          float m = x[r];
#pragma unroll
          for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
          if (lane == 0) tmax[sw * NROW + r] = m;
        }
        named_bar_sync(1, 128);
        float alpha[NROW];
#pragma unroll
        for (int r = 0; r < NROW; ++r) {
          const float tm = fmaxf(fmaxf(tmax[r], tmax[NROW + r]), fmaxf(tmax[2 * NROW + r], tmax[3 * NROW + r]));
          const float mo = m_ref[r];
          const float mn = tm > mo + kRescaleLog2 ? tm : mo;
          alpha[r] = mn == mo ? 1.f : fast_exp2(mo - mn);  // 0 when nothing was seen yet
          psum[r] *= alpha[r];
        }
        named_bar_sync(1, 128);  // everyone has the old reference before it moves
        if (sw == 0) {
          const int r = lane;
          const float tm = fmaxf(fmaxf(tmax[r], tmax[NROW + r]), fmaxf(tmax[2 * NROW + r], tmax[3 * NROW + r]));
          if (tm > m_ref[r] + kRescaleLog2) m_ref[r] = tm;
        }
        if (t > 0) {
          // O^T of the previous tile must be complete before it is rescaled
          okr = warp_wait(&p_free[(t - 1) & 1], ((t - 1) >> 1) & 1, p.wait_ns, abort_flag);
          if (okr) {
            tc_fence_after();
#pragma unroll 1
            for (int mi = 0; mi < C::NMT; ++mi) {
              uint32_t v[32];
              tmem_ld32(t_lane + C::TM_O + mi * NROW, v);
              tmem_ld_wait();
#pragma unroll
              for (int r = 0; r < NROW; ++r) v[r] = __float_as_uint(__uint_as_float(v[r]) * alpha[r]);
              tmem_st32(t_lane + C::TM_O + mi * NROW, v);
            }
            tmem_st_wait();
          }
        }
        if (lane == 0) flags[4 + sw] = okr ? 1 : 0;
        named_bar_sync(1, 128);  // new reference and rescaled O^T visible to all
        if (!(flags[4] & flags[5] & flags[6] & flags[7])) {
          ok = false;
          break;
        }
#pragma unroll
        for (int r = 0; r < NROW; ++r) {
          const float m = m_ref[r];
          mr8[r] = m + kRescaleLog2;
          mrz[r] = m == -INFINITY ? 0.f : m;
        }
      }
      // P^T row of this key (bf16, 32 rows = 64 B) into the 128-byte-swizzled tile
      if (t >= 2 && !warp_wait(&p_free[t & 1], ((t - 2) >> 1) & 1, p.wait_ns, abort_flag)) {
        ok = false;
        if (!*abort_flag) fail();
      }
      if (kt) {
        uint32_t pk[NROW / 2];
#pragma unroll
        for (int e = 0; e < NROW / 2; ++e) {
          const float p0 = fast_exp2(x[2 * e] - mrz[2 * e]);
          const float p1 = fast_exp2(x[2 * e + 1] - mrz[2 * e + 1]);
          psum[2 * e] += p0;
          psum[2 * e + 1] += p1;
          pk[e] = pack_bf16(p0, p1);
        }
        uint8_t* prow = smem + C::OFF_P + (t & 1) * TKY * 128 + kin * 128;
#pragma unroll
        for (int c = 0; c < NROW / 8; ++c)
          *reinterpret_cast<uint4*>(prow + ((c ^ (kin & 7)) * 16)) = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[t & 1]);
    }
    // row sums over all keys: 16 lanes of each warp, then the four warps
#pragma unroll
    for (int r = 0; r < NROW; ++r) {
      float v = kt ? psum[r] : 0.f;
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) tsum[sw * NROW + r] = v;
    }
    if (ok && !warp_wait(&p_free[(ntiles - 1) & 1], ((ntiles - 1) >> 1) & 1, p.wait_ns, abort_flag)) ok = false;
    named_bar_sync(1, 128);
    if (!ok) {
      if (!*abort_flag) fail();
    } else {
      tc_fence_after();
      // thread = value dimension within each 128-dim M-tile; 32 rows per tcgen05.ld
      const int dim = q * 32 + lane;
#pragma unroll 1
      for (int mi = 0; mi < C::NMT; ++mi) {
        uint32_t v[32];
        tmem_ld32(t_lane + C::TM_O + mi * NROW, v);
        tmem_ld_wait();
        for (int r = 0; r < nrows; ++r) {
          const float l = tsum[r] + tsum[NROW + r] + tsum[2 * NROW + r] + tsum[3 * NROW + r];
          const float o = l > 0.f ? __uint_as_float(v[r]) / l : 0.f;
          const size_t orow = out_row(r);
          if (p.nsplit == 1) {
            p.out[orow * D + mi * 128 + dim] = __float2bfloat16_rn(o);
          } else {
            p.ws_o[(orow * p.nsplit + split) * D + mi * 128 + dim] = o;
          }
        }
      }
      if (sw == 0 && lane < nrows) {
        const int r = lane;
        const float l = tsum[r] + tsum[NROW + r] + tsum[2 * NROW + r] + tsum[3 * NROW + r];
        const float lse = l > 0.f ? (m_ref[r] + log2f(l)) * kLn2 : -INFINITY;
        const size_t orow = out_row(r);
        if (p.nsplit == 1) {
          if (p.lse) p.lse[orow] = lse;
        } else {
          p.ws_lse[orow * p.nsplit + split] = lse;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == MMAW) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TM_COLS);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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

bool encode(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
            const cuuint32_t* box) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_tc(const GqaLaunch& a, cudaStream_t stream) {
  using C = TcCfg<D>;
  static std::atomic<unsigned long long> smem_limit_set{0};
  if (cudaError_t e = ensure_smem_limit(gqa_tc_kernel<D>, C::SMEM, smem_limit_set)) return e;
  const uint64_t tokens = a.paged ? (uint64_t)a.num_pages * TKY : (uint64_t)a.b * a.capacity;
  CUtensorMap tq, tk, tv;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)a.b * a.hq * a.s};
    const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    const cuuint32_t box[2] = {64, NROW};
    if (!encode(&tq, a.q, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)a.hkv, tokens};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)a.hkv * D * 2};
    const cuuint32_t box[3] = {64, 1, TKY};
    if (!encode(&tk, a.k, 3, dims, strides, box) || !encode(&tv, a.v, 3, dims, strides, box))
      return cudaErrorInvalidValue;
  }
  TcParams p;
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
  p.nrb = (p.R + NROW - 1) / NROW;
  p.nsplit = a.nsplit;
  p.chunk = a.chunk;
  p.scale_log2 = a.scale * kLog2e;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.lse = a.lse;
  p.ws_o = a.ws_o;
  p.ws_lse = a.ws_lse;
  p.err = a.err;
  p.wait_ns = a.wait_ns;
  dim3 grid(p.nrb * a.nsplit, a.hkv, a.b);
  gqa_tc_kernel<D><<<grid, NTHREADS, C::SMEM, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

bool gqa_tc_eligible(int rows, int d) { return rows > 16 && (d == 128 || d == 256); }
int gqa_tc_rows_per_cta() { return NROW; }

cudaError_t launch_gqa_tc(const GqaLaunch& a, cudaStream_t stream) {
  if (a.d == 128) return launch_tc<128>(a, stream);
  if (a.d == 256) return launch_tc<256>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace decattn
