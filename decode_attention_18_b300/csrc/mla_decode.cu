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
//     is consumed in tiles of 128 latent rows. For S, each tile streams
//     through a ring of 16 KB shared-memory slots, one 64-wide column chunk
//     [128 rows x 64] (or the RoPE chunk) at a time, loaded by TMA as two
//     64-row boxes (so a box never crosses a 64-token page). For O, the
//     CTA's 256 output columns of the same rows stream again (from L2) in
//     16-row slabs through a second ring.
//   * tcgen05.mma (kind::f16, bf16 in, fp32 accumulate in Tensor Memory):
//       S  = Q' K'^T    M=128, N=128 keys, K=k+p  (K-major A and B)
//       O += P Z_half   M=128, N=256,      K=16 keys per slab (Z read MN-major)
//     The fp32 accumulator of 128 rows x k = 512 columns would fill all of
//     TMEM, so the output columns are split over 2 CTAs per row tile, each
//     recomputing S for the same rows; TMEM holds O (256 columns) and two
//     128-column S buffers, so S of the next tile is computed while the
//     softmax of the current one runs. On this part a tcgen05.mma costs about
//     100 cycles to issue whatever its N, so N = 128 keeps the tensor pipe fed.
//   * Softmax warps (thread = row) read S with tcgen05.ld, apply the causal
//     mask and scale, and keep a reference maximum that moves only when a
//     row's maximum grows by more than 2^8 (O is then rescaled in TMEM); P is
//     written as bf16 into shared memory (128-byte swizzled) for the O MMA.
//   * Warp roles: warp 0 issues TMA, warp 1 issues MMAs (one thread) and owns
//     the TMEM allocation, warps 2-5 run the softmax and the epilogue.
//   * Latent rows past the sequence end may hold anything: slabs wholly past
//     it are not loaded or multiplied; the one slab that straddles it has its
//     rows past the end zeroed before the O MMA, so P Z stays finite.
//   * Every mbarrier wait is bounded; on time-out the CTA records the error,
//     stops issuing work, waits for its own copies and MMAs, frees TMEM and
//     returns.
// Output: with a single chunk, bf16 O_lat and the LSE directly; otherwise fp32
// partials (O / l, LSE) merged by the combine kernel.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"

namespace decattn {

namespace {

constexpr int TK = 128;         // latent rows (keys) per S tile
constexpr int NS = 2;           // S-ring slots (one 64-wide column chunk of a tile each)
constexpr int NO = 2;           // O-ring slots (one 16-row slab each)
constexpr int SLAB = 16;        // keys per O slab (= MMA K)
constexpr int BMROWS = 128;     // query rows per CTA (MMA M)
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
  static constexpr int PE_ROW = P * 2;          // bytes per RoPE row
  static constexpr uint32_t PE_SWZ = PE_ROW == 128 ? kSw128 : (PE_ROW == 64 ? kSw64 : kSw32);
  static constexpr int Q_BOX = BMROWS * 128;
  static constexpr int Q_LAT = NBL * Q_BOX;
  static constexpr int Q_PE = BMROWS * PE_ROW;
  static constexpr int S_SLOT = TK * 128;             // one [128 keys x 64] chunk
  static constexpr int HALF_LAT = 64 * 128;           // one 64-row box of a latent chunk
  static constexpr int HALF_PE = 64 * PE_ROW;         // one 64-row box of the RoPE chunk
  static constexpr int O_SUB = SLAB * 128;            // [16 keys x 64 cols]
  static constexpr int O_SLOT = (KLH / 64) * O_SUB;   // [16 keys x KLH cols]
  static constexpr int P_BOX = BMROWS * 128;          // [128 rows x 64 keys] of P
  static constexpr int OFF_QPE = Q_LAT;
  static constexpr int OFF_P = align1024(Q_LAT + Q_PE);
  static constexpr int OFF_SRING = OFF_P + 2 * P_BOX;
  static constexpr int OFF_ORING = OFF_SRING + NS * S_SLOT;
  static constexpr int OFF_BAR = align1024(OFF_ORING + NO * O_SLOT);
  static constexpr int SMEM = OFF_BAR + 256 + 1024;  // + barriers + alignment slack
  static constexpr int TM_S = KLH;                   // two S buffers after the O accumulator
  static constexpr int TM_COLS = pow2_cols(KLH + 2 * TK);
  static_assert(KL % 64 == 0 && KLH % 64 == 0 && KLH <= 256, "latent width");
  static_assert(P % 16 == 0 && PE_ROW <= 128, "rope width");
  static_assert(SMEM <= 232448, "shared memory");
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

template <int KL, int P>
__global__ void __launch_bounds__(192, 1)
    mla_latent_kernel(const __grid_constant__ CUtensorMap tm_qz, const __grid_constant__ CUtensorMap tm_qpe,
                      const __grid_constant__ CUtensorMap tm_z64, const __grid_constant__ CUtensorMap tm_kpe64,
                      const __grid_constant__ CUtensorMap tm_z16, MlaParams p) {
  using C = MlaCfg<KL, P>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const uint32_t sb = smem_u32(smem);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int lh = blockIdx.x % C::NH;
  const int mt = blockIdx.x / C::NH;
  const int split = blockIdx.y;
  const int bi = blockIdx.z;
  const int L = p.seqlens[bi];
  const int kstart = split * p.chunk;
  if (kstart >= L) {  // chunk past the end: the combine skips it
    if (L <= 0 && p.nsplit == 1) {  // empty sequence without a combine pass: zero rows, LSE = -inf
      for (int idx = threadIdx.x; idx < BMROWS * (C::KLH / 8); idx += blockDim.x) {
        const int r = idx / (C::KLH / 8);
        if (mt * BMROWS + r >= p.rows) continue;
        const size_t grow = (size_t)bi * p.rows + mt * BMROWS + r;
        *reinterpret_cast<uint4*>(p.o_lat + grow * KL + lh * C::KLH + (idx % (C::KLH / 8)) * 8) =
            make_uint4(0, 0, 0, 0);
        if (p.lse && lh == 0 && idx % (C::KLH / 8) == 0) p.lse[grow] = -INFINITY;
      }
    }
    return;
  }
  const int kend = min(L, kstart + p.chunk);
  const int ntiles = (kend - kstart + TK - 1) / TK;
  const int qrow0 = bi * p.rows + mt * BMROWS;  // first flattened [b*h*s] query row
  auto tile_keys = [&](int t) { return min(TK, kend - (kstart + t * TK)); };
  auto tile_slabs = [&](int t) { return (tile_keys(t) + SLAB - 1) / SLAB; };

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* s_full = bars + 1;    // [NS]  chunk landed
  uint64_t* s_empty = bars + 3;   // [NS]  chunk consumed by the S MMAs
  uint64_t* o_full = bars + 5;    // [NO]  slab landed
  uint64_t* o_empty = bars + 7;   // [NO]  slab consumed by the O MMA
  uint64_t* s_ready = bars + 9;   // [2]   S tile in TMEM
  uint64_t* p_full = bars + 11;   //       P in shared memory (+ O rescaled)
  uint64_t* o_done = bars + 12;   //       O MMAs of a tile complete
  uint64_t* test_bar = bars + 13;
  uint64_t* fin_bar = bars + 14;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 15);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 16);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < NS; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], 1);
    }
    for (int i = 0; i < NO; ++i) {
      mbar_init(&o_full[i], 1);
      mbar_init(&o_empty[i], 1);
    }
    mbar_init(&s_ready[0], 1);
    mbar_init(&s_ready[1], 1);
    mbar_init(p_full, 4);  // one arrival per softmax warp
    mbar_init(o_done, 1);
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
    prefetch_tmap(&tm_z16);
  }
  if (warp == 1) {
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

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_stream = policy_evict_first();
      const uint64_t pol_keep = policy_evict_last();
      int last_s[NS] = {-1, -1}, last_o[NO] = {-1, -1};
      mbar_expect_tx(q_full, C::Q_LAT + C::Q_PE);
      for (int kb = 0; kb < C::NBL; ++kb) tma_load_2d(sb + kb * C::Q_BOX, &tm_qz, kb * 64, qrow0, q_full);
      tma_load_2d(sb + C::OFF_QPE, &tm_qpe, 0, qrow0, q_full);
      int sc = 0, oc = 0;
      bool ok = true;
      for (int t = 0; ok && t <= ntiles; ++t) {
        if (t < ntiles) {
          const int key0 = kstart + t * TK;
          const int nhalf = tile_keys(t) > 64 ? 2 : 1;
          const int row_a = cache_row(p, bi, key0);
          const int row_b = nhalf > 1 ? cache_row(p, bi, key0 + 64) : 0;
          for (int j = 0; j < C::NCH; ++j, ++sc) {
            const int slot = sc % NS;
            if (sc >= NS && !mbar_wait(&s_empty[slot], ((sc / NS) - 1) & 1, p.wait_ns, abort_flag)) {
              ok = false;
              break;
            }
            const bool pe = j == C::NBL;
            const uint32_t dst = sb + C::OFF_SRING + slot * C::S_SLOT;
            const uint32_t half = pe ? C::HALF_PE : C::HALF_LAT;
            mbar_expect_tx(&s_full[slot], half * nhalf);
            if (pe) {
              tma_load_2d_hint(dst, &tm_kpe64, 0, row_a, &s_full[slot], pol_keep);
              if (nhalf > 1) tma_load_2d_hint(dst + half, &tm_kpe64, 0, row_b, &s_full[slot], pol_keep);
            } else {
              // the CTA's own output half is read again for O (from L2): keep it; the rest streams
              const uint64_t pol = (j / (C::NBL / C::NH)) == lh ? pol_keep : pol_stream;
              tma_load_2d_hint(dst, &tm_z64, j * 64, row_a, &s_full[slot], pol);
              if (nhalf > 1) tma_load_2d_hint(dst + half, &tm_z64, j * 64, row_b, &s_full[slot], pol);
            }
            last_s[slot] = sc;
          }
        }
        if (ok && t >= 1) {
          const int u = t - 1;
          const int key0 = kstart + u * TK;
          const int nsl = tile_slabs(u);
          for (int s = 0; s < nsl; ++s, ++oc) {
            const int slot = oc % NO;
            if (oc >= NO && !mbar_wait(&o_empty[slot], ((oc / NO) - 1) & 1, p.wait_ns, abort_flag)) {
              ok = false;
              break;
            }
            const int row = cache_row(p, bi, key0 + s * SLAB);
            const uint32_t dst = sb + C::OFF_ORING + slot * C::O_SLOT;
            mbar_expect_tx(&o_full[slot], C::O_SLOT);
            for (int i = 0; i < C::KLH / 64; ++i)
              tma_load_2d_hint(dst + i * C::O_SUB, &tm_z16, lh * C::KLH + i * 64, row, &o_full[slot], pol_stream);
            last_o[slot] = oc;
          }
        }
      }
      if (!ok && !*abort_flag) fail();
      // no copy may still be landing in shared memory when the CTA exits
      mbar_wait(q_full, 0, kTeardownNs, nullptr);
      for (int i = 0; i < NS; ++i)
        if (last_s[i] >= 0) mbar_wait(&s_full[i], (last_s[i] / NS) & 1, kTeardownNs, nullptr);
      for (int i = 0; i < NO; ++i)
        if (last_o[i] >= 0) mbar_wait(&o_full[i], (last_o[i] / NO) & 1, kTeardownNs, nullptr);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (lane 0; the warp zeroes tails)
    bool ok = true;
    if (lane == 0) {
      if (p.test_timeout && !mbar_wait(test_bar, 0, kTestWaitNs, abort_flag)) ok = false;
      if (ok && !mbar_wait(q_full, 0, p.wait_ns, abort_flag)) ok = false;
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    tc_fence_after();
    constexpr uint32_t idS = idesc_bf16_f32(BMROWS, TK, false, false);
    constexpr uint32_t idO = idesc_bf16_f32(BMROWS, C::KLH, false, true);
    int sc = 0, oc = 0;
    for (int t = 0; ok && t <= ntiles; ++t) {
      if (t < ntiles) {
        const uint32_t d_s = tmem + C::TM_S + (t & 1) * TK;
        for (int j = 0; j < C::NCH; ++j, ++sc) {
          const int slot = sc % NS;
          if (lane == 0) {
            if (!mbar_wait(&s_full[slot], (sc / NS) & 1, p.wait_ns, abort_flag)) {
              ok = false;
            } else {
              tc_fence_after();
              const uint32_t src = sb + C::OFF_SRING + slot * C::S_SLOT;
              if (j < C::NBL) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  tc_mma_ss(d_s, smem_desc(sb + j * C::Q_BOX + kk * 32, 16, 1024, kSw128),
                            smem_desc(src + kk * 32, 16, 1024, kSw128), idS, (j > 0 || kk > 0) ? 1u : 0u);
              } else {
#pragma unroll
                for (int kk = 0; kk < P / 16; ++kk)
                  tc_mma_ss(d_s, smem_desc(sb + C::OFF_QPE + kk * 32, 16, 8 * C::PE_ROW, C::PE_SWZ),
                            smem_desc(src + kk * 32, 16, 8 * C::PE_ROW, C::PE_SWZ), idS, 1u);
              }
              tc_commit(&s_empty[slot]);
            }
          }
          if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
            ok = false;
            break;
          }
        }
        if (!ok) break;
        if (lane == 0) tc_commit(&s_ready[t & 1]);
      }
      if (t >= 1) {
        const int u = t - 1;
        const int key0 = kstart + u * TK;
        const int nsl = tile_slabs(u);
        if (lane == 0 && !mbar_wait(p_full, u & 1, p.wait_ns, abort_flag)) ok = false;
        if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
          ok = false;
          break;
        }
        for (int s = 0; s < nsl; ++s, ++oc) {
          const int slot = oc % NO;
          if (lane == 0 && !mbar_wait(&o_full[slot], (oc / NO) & 1, p.wait_ns, abort_flag)) ok = false;
          if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
            ok = false;
            break;
          }
          __syncwarp();
          const int first_bad = L - (key0 + s * SLAB);  // rows at or past the sequence end
          if (first_bad < SLAB) {
            const uint32_t base = C::OFF_ORING + slot * C::O_SLOT;
            const int nrow = SLAB - first_bad;
            for (int idx = lane; idx < nrow * (C::KLH / 64) * 8; idx += 32) {
              const int rr = first_bad + idx / ((C::KLH / 64) * 8);
              const int rem = idx % ((C::KLH / 64) * 8);
              *reinterpret_cast<uint4*>(smem + base + (rem / 8) * C::O_SUB + rr * 128 + (rem % 8) * 16) =
                  make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            __syncwarp();
          }
          if (lane == 0) {
            tc_fence_after();
            const uint64_t a = smem_desc(sb + C::OFF_P + (s / 4) * C::P_BOX + (s % 4) * 32, 16, 1024, kSw128);
            // Z slab read MN-major: 64-column boxes O_SUB apart, 8-key groups 1024 B apart
            const uint64_t bd = smem_desc(sb + C::OFF_ORING + slot * C::O_SLOT, C::O_SUB, 1024, kSw128);
            tc_mma_ss(tmem, a, bd, idO, (u > 0 || s > 0) ? 1u : 0u);
            tc_commit(&o_empty[slot]);
          }
        }
        if (!ok) break;
        if (lane == 0) tc_commit(o_done);
      }
    }
    if (lane == 0) {
      if (!ok && !*abort_flag) fail();
      // every issued tcgen05 operation has finished before TMEM is released
      tc_commit(fin_bar);
      mbar_wait(fin_bar, 0, kTeardownNs, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int r = q * 32 + lane;
    const int row_in_seq = mt * BMROWS + r;
    const bool row_ok = row_in_seq < p.rows;
    const int lim = row_ok ? min(kend, L - p.s + (row_in_seq % p.s) + 1) : 0;  // exclusive key limit
    const uint32_t t_lane = tmem + ((uint32_t)(q * 32) << 16);
    float m_ref = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      // waits are made warp-uniform: the tcgen05 loads below are warp-collective
      if (!__all_sync(0xffffffffu, mbar_wait(&s_ready[t & 1], (t >> 1) & 1, p.wait_ns, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int key0 = kstart + t * TK;
      float x[TK];
      float mx = -INFINITY;
#pragma unroll
      for (int c0 = 0; c0 < TK; c0 += 32) {
        uint32_t sv[32];
        tmem_ld32(t_lane + C::TM_S + (t & 1) * TK + c0, sv);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float v = (key0 + c0 + c < lim) ? __uint_as_float(sv[c]) * p.scale_log2 : -INFINITY;
          x[c0 + c] = v;
          mx = fmaxf(mx, v);
        }
      }
      // the previous O MMAs must be complete: they still read P, and O may be rescaled
      if (t > 0 && !__all_sync(0xffffffffu, mbar_wait(o_done, (t - 1) & 1, p.wait_ns, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      float alpha = 1.f;
      if (mx > m_ref + kRescaleLog2) {
        alpha = exp2f(m_ref - mx);  // 0 when nothing was seen yet
        m_ref = mx;
        l_run *= alpha;
      }
      if (t > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        for (int c0 = 0; c0 < C::KLH; c0 += 32) {
          uint32_t v[32];
          tmem_ld32(t_lane + c0, v);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * alpha);
          tmem_st32(t_lane + c0, v);
        }
        tmem_st_wait();
      }
      // P row (bf16) into two 128-byte-swizzled [128 rows x 64 keys] boxes
      float ps = 0.f;
      const bool live = m_ref != -INFINITY;
#pragma unroll
      for (int ch = 0; ch < TK / 8; ++ch) {
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p0 = live ? exp2f(x[ch * 8 + 2 * e] - m_ref) : 0.f;
          const float p1 = live ? exp2f(x[ch * 8 + 2 * e + 1] - m_ref) : 0.f;
          ps += p0 + p1;
          pk[e] = pack_bf16(p0, p1);
        }
        const int box = ch / 8, lc = ch % 8;
        *reinterpret_cast<uint4*>(smem + C::OFF_P + box * C::P_BOX + r * 128 + ((lc ^ (r & 7)) * 16)) =
            make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
      l_run += ps;
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    if (ok && !__all_sync(0xffffffffu, mbar_wait(o_done, (ntiles - 1) & 1, p.wait_ns, abort_flag))) ok = false;
    if (!ok) {
      if (!*abort_flag) fail();
    } else {
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      const float lse = l_run > 0.f ? (m_ref + log2f(l_run)) * kLn2 : -INFINITY;
      const size_t grow = (size_t)qrow0 + r;
      for (int c0 = 0; c0 < C::KLH; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(t_lane + c0, v);
        tmem_ld_wait();
        if (!row_ok) continue;
        const int col = lh * C::KLH + c0;
        if (p.nsplit == 1) {
          uint4* dst = reinterpret_cast<uint4*>(p.o_lat + grow * KL + col);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[e] = make_uint4(pack_bf16(__uint_as_float(v[8 * e + 0]) * inv, __uint_as_float(v[8 * e + 1]) * inv),
                                pack_bf16(__uint_as_float(v[8 * e + 2]) * inv, __uint_as_float(v[8 * e + 3]) * inv),
                                pack_bf16(__uint_as_float(v[8 * e + 4]) * inv, __uint_as_float(v[8 * e + 5]) * inv),
                                pack_bf16(__uint_as_float(v[8 * e + 6]) * inv, __uint_as_float(v[8 * e + 7]) * inv));
        } else {
          float4* dst = reinterpret_cast<float4*>(p.ws_o + (grow * p.nsplit + split) * KL + col);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            dst[e] = make_float4(__uint_as_float(v[4 * e + 0]) * inv, __uint_as_float(v[4 * e + 1]) * inv,
                                 __uint_as_float(v[4 * e + 2]) * inv, __uint_as_float(v[4 * e + 3]) * inv);
        }
      }
      if (row_ok && lh == 0) {
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
    tmem_dealloc(tmem, C::TM_COLS);
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
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(mla_latent_kernel<KL, P>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  const uint64_t qrows = (uint64_t)a.b * a.h * a.s;
  const uint64_t krows = a.paged ? (uint64_t)a.num_pages * 64 : (uint64_t)a.b * a.capacity;
  CUtensorMap tqz, tqpe, tz64, tkpe64, tz16;
  if (!make_map(&tqz, a.qz, qrows, KL, BMROWS, 64) || !make_map(&tqpe, a.q_pe, qrows, P, BMROWS, P) ||
      !make_map(&tz64, a.z, krows, KL, 64, 64) || !make_map(&tkpe64, a.k_pe, krows, P, 64, P) ||
      !make_map(&tz16, a.z, krows, KL, SLAB, 64))
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
  dim3 grid(C::NH * mtiles, a.nsplit, a.b);
  mla_latent_kernel<KL, P><<<grid, 192, C::SMEM, stream>>>(tqz, tqpe, tz64, tkpe64, tz16, p);
  return cudaGetLastError();
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
