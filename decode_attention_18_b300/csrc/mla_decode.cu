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
// Kernel design (one CTA = 128 query rows x one context chunk x one latent
// partition of the output):
//   * All h*s query rows of a sequence are packed into the MMA M dimension
//     (row = head*s + token), 128 rows per CTA.
//   * Q' = [Qz | q_pe] stays in shared memory for the whole chunk; tiles of 32
//     latent rows [Z | K_pe] stream from HBM once per CTA through a 2-stage
//     TMA pipeline (128-byte swizzled boxes, evict-first L2 policy).
//   * tcgen05.mma (kind::f16, bf16 in, fp32 accumulate in Tensor Memory):
//       S  = Q' K'^T           M=128, N=32, K=k+p   (K-major A and B)
//       O += P Z_part          M=128, N=k/NH, K=32  (Z read MN-major: the very
//                                                    same shared tile as above)
//     S is double-buffered in TMEM; the fp32 O accumulator of a 128-row tile
//     is 128 x k, which for k = 512 fills all 512 TMEM columns, so the output
//     columns are split over NH = 2 CTAs (each recomputes S for its rows).
//   * Softmax warps (thread = row) read S with tcgen05.ld, apply the causal
//     mask and scale, and keep a running reference maximum that moves only
//     when a row's maximum grows by more than 2^8 (then O is rescaled in
//     TMEM); P (bf16) goes to shared memory for the second MMA.
//   * Warp roles: warp 0 issues TMA, warp 1 issues MMAs (one thread) and owns
//     the TMEM allocation, warps 2-5 run the softmax and the epilogue.
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

constexpr int TK = 32;          // latent rows (keys) per tile
constexpr int NSTAGE = 2;
constexpr int BMROWS = 128;     // query rows per CTA (MMA M)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.f;                      // move the reference max only past 2^8
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
  static constexpr int NH = KL >= 512 ? 2 : 1;  // CTAs per 128-row tile (output-column partitions)
  static constexpr int KLH = KL / NH;           // O columns per CTA
  static constexpr int NBL = KL / 64;           // 64-wide (128-byte) latent boxes
  static constexpr int PE_ROW = P * 2;          // bytes per RoPE row
  static constexpr uint32_t PE_SWZ = PE_ROW == 128 ? kSw128 : (PE_ROW == 64 ? kSw64 : kSw32);
  static constexpr int Q_BOX = BMROWS * 128;
  static constexpr int Q_LAT = NBL * Q_BOX;
  static constexpr int Q_PE = BMROWS * PE_ROW;
  static constexpr int KV_BOX = TK * 128;
  static constexpr int KV_LAT = NBL * KV_BOX;
  static constexpr int KV_PE = TK * PE_ROW;
  static constexpr int STAGE = align1024(KV_LAT + KV_PE);
  static constexpr int P_BYTES = BMROWS * TK * 2;  // P tile, rows of 64 B (64-byte swizzle)
  static constexpr int OFF_QPE = Q_LAT;
  static constexpr int OFF_STAGE = align1024(Q_LAT + Q_PE);
  static constexpr int OFF_P = OFF_STAGE + NSTAGE * STAGE;
  static constexpr int OFF_BAR = OFF_P + P_BYTES;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;  // + barriers + alignment slack
  static constexpr int TM_S = KLH;                   // S buffers after the O accumulator
  static constexpr int TM_COLS = pow2_cols(KLH + NSTAGE * TK);
  static_assert(KL % 64 == 0 && KLH % 32 == 0 && KLH <= 256, "latent width");
  static_assert(P % 16 == 0 && PE_ROW <= 128, "rope width");
  static_assert(SMEM <= 232448, "shared memory");
};

template <int KL, int P>
__global__ void __launch_bounds__(192, 1)
    mla_latent_kernel(const __grid_constant__ CUtensorMap tm_qz, const __grid_constant__ CUtensorMap tm_qpe,
                      const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_kpe,
                      MlaParams p) {
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

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* kv_full = bars + 1;   // [NSTAGE]
  uint64_t* kv_empty = bars + 3;  // [NSTAGE]
  uint64_t* s_full = bars + 5;    // [NSTAGE]
  uint64_t* s_free = bars + 7;    // [NSTAGE]
  uint64_t* p_full = bars + 9;
  uint64_t* o_done = bars + 10;
  uint64_t* test_bar = bars + 11;
  uint64_t* fin_bar = bars + 12;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 13);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 14);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int st = 0; st < NSTAGE; ++st) {
      mbar_init(&kv_full[st], 1);
      mbar_init(&kv_empty[st], 1);
      mbar_init(&s_full[st], 1);
      mbar_init(&s_free[st], 4);  // one arrival per softmax warp
    }
    mbar_init(p_full, 4);
    mbar_init(o_done, 1);
    mbar_init(test_bar, 1);  // never signalled: the forced-timeout test waits on it
    mbar_init(fin_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_qz);
    prefetch_tmap(&tm_qpe);
    prefetch_tmap(&tm_z);
    prefetch_tmap(&tm_kpe);
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
      int last_issued[NSTAGE] = {-1, -1};
      mbar_expect_tx(q_full, C::Q_LAT + C::Q_PE);
      for (int kb = 0; kb < C::NBL; ++kb) tma_load_2d(sb + kb * C::Q_BOX, &tm_qz, kb * 64, qrow0, q_full);
      tma_load_2d(sb + C::OFF_QPE, &tm_qpe, 0, qrow0, q_full);
      for (int t = 0; t < ntiles; ++t) {
        const int st = t % NSTAGE;
        if (t >= NSTAGE && !mbar_wait(&kv_empty[st], ((t / NSTAGE) - 1) & 1, p.wait_ns, abort_flag)) {
          if (!*abort_flag) fail();
          break;
        }
        if (*abort_flag) break;
        const int key0 = kstart + t * TK;
        int row;
        if (p.paged) {
          int page = p.block_table[(size_t)bi * p.max_pages + key0 / 64];
          if (page < 0 || page >= p.num_pages) {
            raise_error(p.err, kErrBadPage);
            page = 0;  // stay inside the pool; the result is flagged invalid
          }
          row = page * 64 + (key0 % 64);
        } else {
          row = bi * p.capacity + key0;
        }
        const uint32_t dst = sb + C::OFF_STAGE + st * C::STAGE;
        mbar_expect_tx(&kv_full[st], C::KV_LAT + C::KV_PE);
        for (int kb = 0; kb < C::NBL; ++kb)
          tma_load_2d_hint(dst + kb * C::KV_BOX, &tm_z, kb * 64, row, &kv_full[st], pol_stream);
        tma_load_2d_hint(dst + C::KV_LAT, &tm_kpe, 0, row, &kv_full[st], pol_stream);
        last_issued[st] = t;
      }
      // no copy may still be landing in shared memory when the CTA exits
      mbar_wait(q_full, 0, kTeardownNs, nullptr);
      for (int st = 0; st < NSTAGE; ++st)
        if (last_issued[st] >= 0) mbar_wait(&kv_full[st], (last_issued[st] / NSTAGE) & 1, kTeardownNs, nullptr);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = true;
      if (p.test_timeout && !mbar_wait(test_bar, 0, kTestWaitNs, abort_flag)) {
        fail();
        ok = false;
      }
      if (ok && !mbar_wait(q_full, 0, p.wait_ns, abort_flag)) {
        fail();
        ok = false;
      }
      tc_fence_after();
      constexpr uint32_t idS = idesc_bf16_f32(BMROWS, TK, false, false);
      constexpr uint32_t idO = idesc_bf16_f32(BMROWS, C::KLH, false, true);
      for (int t = 0; ok && t <= ntiles; ++t) {
        if (t < ntiles) {
          const int st = t % NSTAGE;
          if (!mbar_wait(&kv_full[st], (t / NSTAGE) & 1, p.wait_ns, abort_flag) ||
              (t >= NSTAGE && !mbar_wait(&s_free[st], ((t - NSTAGE) / NSTAGE) & 1, p.wait_ns, abort_flag))) {
            if (!*abort_flag) fail();
            break;
          }
          tc_fence_after();
          const uint32_t stage = sb + C::OFF_STAGE + st * C::STAGE;
          const uint32_t d_s = tmem + C::TM_S + st * TK;
          uint32_t acc = 0;
          for (int kb = 0; kb < C::NBL; ++kb) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t a = smem_desc(sb + kb * C::Q_BOX + kk * 32, 16, 1024, kSw128);
              const uint64_t bd = smem_desc(stage + kb * C::KV_BOX + kk * 32, 16, 1024, kSw128);
              tc_mma_ss(d_s, a, bd, idS, acc);
              acc = 1;
            }
          }
#pragma unroll
          for (int kk = 0; kk < P / 16; ++kk) {
            const uint64_t a = smem_desc(sb + C::OFF_QPE + kk * 32, 16, 8 * C::PE_ROW, C::PE_SWZ);
            const uint64_t bd = smem_desc(stage + C::KV_LAT + kk * 32, 16, 8 * C::PE_ROW, C::PE_SWZ);
            tc_mma_ss(d_s, a, bd, idS, 1);
          }
          tc_commit(&s_full[st]);
        }
        if (t >= 1) {
          const int u = t - 1;
          const int su = u % NSTAGE;
          if (!mbar_wait(p_full, u & 1, p.wait_ns, abort_flag)) {
            if (!*abort_flag) fail();
            break;
          }
          tc_fence_after();
          const uint32_t zpart = sb + C::OFF_STAGE + su * C::STAGE + (lh * C::KLH / 64) * C::KV_BOX;
#pragma unroll
          for (int kk = 0; kk < TK / 16; ++kk) {
            const uint64_t a = smem_desc(sb + C::OFF_P + kk * 32, 16, 512, kSw64);
            // Z tile read MN-major: 64-column boxes KV_BOX apart, 8-key groups 1024 B apart
            const uint64_t bd = smem_desc(zpart + kk * 16 * 128, C::KV_BOX, 1024, kSw128);
            tc_mma_ss(tmem, a, bd, idO, (u > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(o_done);
          tc_commit(&kv_empty[su]);
        }
      }
      // every issued tcgen05 operation has finished before TMEM is released
      tc_commit(fin_bar);
      mbar_wait(fin_bar, 0, kTeardownNs, nullptr);
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int r = q * 32 + lane;
    const int row_in_seq = mt * BMROWS + r;
    const bool row_ok = row_in_seq < p.rows;
    const int lim = row_ok ? min(kend, L - p.s + (row_in_seq % p.s) + 1) : 0;  // exclusive key limit
    const uint32_t t_lane = tmem + ((uint32_t)(q * 32) << 16);
    const int sm_tid = threadIdx.x - 64;  // 0..127
    float m_ref = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      const int st = t % NSTAGE;
      // waits are made warp-uniform: the tcgen05 loads below are warp-collective
      if (!__all_sync(0xffffffffu, mbar_wait(&s_full[st], (t / NSTAGE) & 1, p.wait_ns, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sv[32];
      tmem_ld32(t_lane + C::TM_S + st * TK, sv);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[st]);

      const int key0 = kstart + t * TK;
      float x[32];
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        x[c] = (key0 + c < lim) ? __uint_as_float(sv[c]) * p.scale_log2 : -INFINITY;
        mx = fmaxf(mx, x[c]);
      }
      // the previous O MMA must be complete: it still reads P, and O may be rescaled
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
      // latent rows past the sequence end may hold anything: zero them so P Z stays finite
      if (key0 + TK > L) {
        const int first = max(0, L - key0);
        const uint32_t zpart = C::OFF_STAGE + st * C::STAGE + (lh * C::KLH / 64) * C::KV_BOX;
        const int nrow = TK - first;
        for (int idx = sm_tid; idx < nrow * (C::KLH / 64) * 8; idx += 128) {
          const int rr = first + idx / ((C::KLH / 64) * 8);
          const int rem = idx % ((C::KLH / 64) * 8);
          const int box = rem / 8, ch = rem % 8;
          *reinterpret_cast<uint4*>(smem + zpart + box * C::KV_BOX + rr * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      // P row (bf16), 64-byte swizzled K-major layout
      uint32_t pk[16];
      float ps = 0.f;
#pragma unroll
      for (int c = 0; c < 32; c += 2) {
        const float p0 = m_ref == -INFINITY ? 0.f : exp2f(x[c] - m_ref);
        const float p1 = m_ref == -INFINITY ? 0.f : exp2f(x[c + 1] - m_ref);
        pk[c / 2] = pack_bf16(p0, p1);
        ps += p0 + p1;
      }
      l_run += ps;
      uint8_t* prow = smem + C::OFF_P + r * 64;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        const int phys = ch ^ ((r >> 1) & 3);
        *reinterpret_cast<uint4*>(prow + phys * 16) = make_uint4(pk[ch * 4], pk[ch * 4 + 1], pk[ch * 4 + 2], pk[ch * 4 + 3]);
      }
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
  CUtensorMap tqz, tqpe, tz, tkpe;
  if (!make_map(&tqz, a.qz, qrows, KL, BMROWS, 64) || !make_map(&tqpe, a.q_pe, qrows, P, BMROWS, P) ||
      !make_map(&tz, a.z, krows, KL, TK, 64) || !make_map(&tkpe, a.k_pe, krows, P, TK, P))
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
  mla_latent_kernel<KL, P><<<grid, 192, C::SMEM, stream>>>(tqz, tqpe, tz, tkpe, p);
  return cudaGetLastError();
}

}  // namespace

int mla_latent_parts(int k) { return k >= 512 ? 2 : 1; }
bool mla_supported(int k, int p) { return (k == 512 && p == 64) || (k == 64 && p == 16); }

cudaError_t launch_mla_latent(const MlaLaunch& a, cudaStream_t stream) {
  if (a.k == 512 && a.p == 64) return launch_kl<512, 64>(a, stream);
  if (a.k == 64 && a.p == 16) return launch_kl<64, 16>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace decattn
