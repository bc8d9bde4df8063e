// Grouped-head split-KV decode attention (MHA / GQA / MQA) for sm_103a.
//
// Follows the grouped-head rows of the summary table in "Why MLA and MTP
// Fight Each Other" (MHA, GQA, MQA are one computation with different KV-head
// counts), the "MHA vs GQA" Q&A section 1 (a KV head serves Hq/Hkv query
// heads) and the contiguous grouping of the "MQA, GQA & MLA" lesson.
//
// One CTA takes one (sequence, KV head, context chunk, block of query rows).
// The query rows of a KV head are its G = Hq/Hkv query heads times the s new
// tokens (row = head_in_group * s + token), so every K/V byte fetched from HBM
// serves all G*s rows: the kernel is bound by the cache read (AI ~ G).
//
//  * K/V tiles of 64 keys stream through a 3-4 stage pipeline of TMA copies:
//    one thread requests each tile of K and of V as [64 tokens x 64 dims] boxes
//    of a 3-D tensor map (tokens, KV heads, d), landing 128-byte swizzled in
//    shared memory and completing on the stage's mbarrier.
//  * 4 warps per 16-row m-tile (MT m-tiles, 128*MT threads); each warp owns 16
//    keys of a tile: S = Q K^T and O += P V run on mma.sync m16n8k16 (bf16 in,
//    fp32 accumulate); the score fragment is reused in registers as the A
//    operand of P V.
//  * Online softmax per warp with quad shuffles (exp2 domain); the four key
//    slices of an m-tile are merged through shared memory at the end.
//  * Output: with one chunk, bf16 rows and the LSE directly; otherwise fp32
//    (O, LSE) partials for the combine kernel.
//  * Every kernel here is launched as a programmatic dependent of the kernel
//    before it on the stream and waits for it (griddepcontrol.wait) before its
//    first global read, so launch and block scheduling overlap that kernel's end.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"

namespace decattn {

namespace {

struct GqaParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const int32_t* seqlens;
  const int32_t* block_table;
  int max_pages, paged, capacity, num_pages;
  int b, s, hq, hkv, G, R, nrb, nsplit, chunk;
  float scale_log2;
  __nv_bfloat16* out;
  float* lse;
  float* ws_o;
  float* ws_lse;
  int* meta;  // balanced mode: per work item {first partial record, record count}
  unsigned* err;
  unsigned long long wait_ns;  // limit of the tile waits
  int test_timeout;            // nonzero: the first tile wait also waits on a barrier nothing signals
  float v_scale;               // FP8 cache: value dequantisation scale, applied to the output (else 1)
};

constexpr int kTileKeys = 64;
constexpr int kTileBlk = kTileKeys * 128;  // one [64 keys x 128 bytes] block of a tile (64 bf16 dims or 128 E4M3)
constexpr int kSlices = 4;  // warps (key slices of 16) per m-tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.f;  // move a row's reference maximum only past 2^8
constexpr unsigned long long kTeardownNs = 1000000000ull;  // 1 s for own copies after a time-out
constexpr unsigned long long kTestWaitNs = 1000000ull;     // 1 ms forced-timeout wait

// DK: width of a query / key row; DV: width of a value / output row (equal for plain
// grouped-head attention; 192 and 128 for the expanded MLA form, whose keys carry the
// 64 RoPE dimensions that its values lack).
template <int DK, int DV, int MT_, bool FP8_ = false>
struct GqaCfg {
  static constexpr bool FP8 = FP8_;  // cache in e4m3 bytes
  // FP8 with 128-byte (or longer) rows: byte tiles land 128-byte swizzled and are widened
  // in registers after ldmatrix (f16 MMAs); with 64-byte rows they are widened to a bf16
  // work tile in shared memory each tile
  static constexpr bool REG8 = FP8_ && DK >= 128;
  static constexpr int MT = MT_;  // 16-row m-tiles per CTA
  static constexpr int THREADS = 128 * MT;
  static constexpr int K_TILE = kTileKeys * DK * 2;  // one K tile (bf16, as the MMAs read it)
  static constexpr int V_TILE = kTileKeys * DV * 2;  // one V tile
  static constexpr int CACHE_ELEM = FP8 ? 1 : 2;     // bytes per cached value
  static constexpr int K_LOAD = kTileKeys * DK * CACHE_ELEM;  // bytes one K tile copy lands
  static constexpr int V_LOAD = kTileKeys * DV * CACHE_ELEM;
  static constexpr int STAGE_BYTES = K_LOAD + V_LOAD;
  // pipeline stages: 4 for small rows, 3 for 128 or 256 dims (two resp. one CTA per SM);
  // the 192/128 form takes 4 (160 KB, one CTA per SM, three tiles in flight); an FP8
  // stage is half as large, so it takes twice as many stages in the same space
  static constexpr int NST = REG8 ? 6 : (FP8 ? (DK <= 64 ? 6 : 4) : ((DK <= 64 || DK != DV) ? 4 : 3));
  // FP8 with a work tile: the bf16 tile pair the MMAs read, written from the landed stage
  static constexpr int WORK_OFF = NST * STAGE_BYTES;
  static constexpr int PIPE_BYTES = NST * STAGE_BYTES + ((FP8 && !REG8) ? K_TILE + V_TILE : 0);
  static constexpr int OSTR = DV + 2;  // padded fp32 row stride of the merge buffer
  static constexpr int RED_BYTES = kSlices * 16 * MT * OSTR * 4;
  static constexpr int SMEM = PIPE_BYTES > RED_BYTES ? PIPE_BYTES : RED_BYTES;
  static_assert(DK % 64 == 0 && DV % 64 == 0, "tiles are 64-dim blocks");
};

// Two e4m3 values (low byte first) to a bf16 pair (low half first). Exact: every e4m3
// value, subnormals included, is a float16 and a bfloat16 value.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint16_t v) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(v), __NV_E4M3);
  __half_raw lo, hi;
  lo.x = h.x;
  hi.x = h.y;
  return pack_bf16(__half2float(__half(lo)), __half2float(__half(hi)));
}

// Shared-memory offset of 16-byte chunk u (16 values) of key row r in a byte tile of
// [64 keys x 128 bytes] blocks, 128-byte swizzled (as TMA writes it)
__device__ __forceinline__ uint32_t tile8_off(int r, int u) {
  return (uint32_t)((u >> 3) * (kTileKeys * 128) + r * 128 + (((u & 7) ^ (r & 7)) << 4));
}

// Shared-memory offset of 16-byte chunk c (8 dims) of key row r in a K or V tile: the
// tile is DK/64 (K) or DV/64 (V) blocks of [64 keys x 128 bytes], each with the 128-byte swizzle (chunk
// index XOR row mod 8) that TMA writes and that keeps ldmatrix free of bank conflicts.
__device__ __forceinline__ uint32_t tile_off(int r, int c) {
  return (uint32_t)((c >> 3) * (kTileKeys * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// Where a segment's result goes.
enum SegOut { kSegFinal = 0, kSegSplit = 1, kSegRecord = 2 };

// Attention of the query rows of block rb of KV head g of sequence bi over keys
// [kstart, kend) (kstart < kend <= L). Query and key rows are DK wide, value and
// output rows DV wide. out_mode kSegFinal writes bf16 rows and the
// LSE; kSegSplit writes fp32 partials at chunk index `slot` of the [row][nsplit]
// layout; kSegRecord writes partial record `slot` ([record][16*MT rows][DV]) of the
// balanced schedule. The caller's threads all enter; shared memory is free again
// when it returns. Returns false (in every thread) when a tile wait ran out: the
// error is recorded, the copies already requested have been waited for (bounded) and
// nothing was written. FP8: the cache holds e4m3 bytes; each landed tile is widened
// to bf16 (exactly) into one work tile pair that the MMAs read; the key scale is part
// of p.scale_log2 and the value scale p.v_scale multiplies the output.
template <int DK, int DV, int MT, bool FP8 = false>
__device__ __forceinline__ bool gqa_segment(const GqaParams& p, const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                            uint64_t* full, uint64_t* never, uint32_t& phase, uint8_t* smem,
                                            float (*s_m)[kSlices][16], float (*s_l)[kSlices][16], int bi, int g,
                                            int rb, int L, int kstart, int kend, int out_mode, int slot) {
  using C = GqaCfg<DK, DV, MT, FP8>;
  constexpr int NT = DV / 8;   // n-tiles of the output
  constexpr int KS = DK / 16;  // k-steps of QK^T
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int mt = warp / kSlices;     // m-tile of this warp
  const int slice = warp % kSlices;  // 16-key slice of each tile
  const int ntiles = (kend - kstart + kTileKeys - 1) / kTileKeys;
  const int mrow0 = (rb * MT + mt) * 16;  // first row (within the KV head's rows) of this warp's m-tile

  // ---- query fragments (A operand; rows past R are zero) and per-row key limits
  uint32_t qa[KS][4];
  int lim[2];
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    const int r = mrow0 + (lane >> 2) + h2 * 8;
    lim[h2] = r < p.R ? min(kend, L - p.s + (r % p.s) + 1) : 0;
  }
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int r = mrow0 + (lane >> 2) + (e & 1) * 8;
      // REG8: the k index of the fragment is permuted to match the byte tiles' ldmatrix
      // layout (fragment k 2c+i is dimension 4c+i, k 2c+8+i is dimension 4c+2+i)
      const int col = C::REG8 ? ks * 16 + (lane & 3) * 4 + (e >> 1) * 2 : ks * 16 + (lane & 3) * 2 + (e >> 1) * 8;
      uint32_t val = 0;
      if (r < p.R) {
        const int j = g * p.G + r / p.s;
        const size_t off = ((size_t)(bi * p.hq + j) * p.s + (r % p.s)) * DK + col;
        val = __ldg(reinterpret_cast<const unsigned int*>(p.q + off));
        if constexpr (C::REG8) val = pack_f16(bf16_lo(val), bf16_hi(val));  // f16 operands
      }
      qa[ks][e] = val;
    }
  }

  // ---- K/V tiles by TMA. Thread 0 requests tile t of this KV head's K and V as DK/64
  // and DV/64 boxes of [64 tokens x 64 dims] (3-D tensor maps over [tokens, KV heads, d]),
  // completing on the stage's mbarrier; every thread waits on it (bounded). For a paged
  // cache the tile is one page. Rows past the segment's end are read as they are (or as
  // zeros past the tensor) and made harmless below.
  const uint32_t sbase = smem_u32(smem);
  // block-table entry of tile t (read one tile ahead of its copy by thread 0)
  auto page_of = [&](int t) -> int {
    if (!p.paged || t >= ntiles) return 0;
    return __ldg(p.block_table + (size_t)bi * p.max_pages + (kstart + t * kTileKeys) / kTileKeys);
  };
  auto issue = [&](int t, int stage, int page) {
    const int key0 = kstart + t * kTileKeys;
    int row0;  // token row of the tile's first key in the cache tensor
    if (p.paged) {
      if (page < 0 || page >= p.num_pages) {
        raise_error(p.err, kErrBadPage);
        page = 0;  // stay inside the pool; the result is flagged invalid
      }
      row0 = page * kTileKeys;
    } else {
      row0 = bi * p.capacity + key0;
    }
    const uint32_t kdst = sbase + stage * C::STAGE_BYTES;
    fence_proxy_async_smem();  // this thread's view: earlier generic writes to the stage come first
    mbar_expect_tx(&full[stage], C::STAGE_BYTES);
    if constexpr (C::REG8) {  // [64 tokens x 128 bytes] boxes, 128-byte swizzle
#pragma unroll
      for (int kb = 0; kb < DK / 128; ++kb) tma_load_3d(kdst + kb * kTileBlk, tm_k, kb * 128, g, row0, &full[stage]);
#pragma unroll
      for (int kb = 0; kb < DV / 128; ++kb)
        tma_load_3d(kdst + C::K_LOAD + kb * kTileBlk, tm_v, kb * 128, g, row0, &full[stage]);
    } else if constexpr (FP8) {  // one unswizzled box each: [64 tokens x DK bytes], [64 tokens x DV bytes]
      tma_load_3d(kdst, tm_k, 0, g, row0, &full[stage]);
      tma_load_3d(kdst + C::K_LOAD, tm_v, 0, g, row0, &full[stage]);
    } else {
      tma_load_4d(kdst, tm_k, 0, row0, 0, g, &full[stage]);
      tma_load_4d(kdst + C::K_TILE, tm_v, 0, row0, 0, g, &full[stage]);
    }
  };

  // ---- online-softmax state and output accumulator (rows lane/4 and lane/4 + 8)
  float o[NT][4];
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;

  // every thread has finished with the shared memory the first copies overwrite (the
  // caller's barrier), so thread 0 can start the pipeline
  int page_next = 0;  // thread 0: block-table entry of the next tile to request
  if (tid == 0) {
#pragma unroll
    for (int t = 0; t < C::NST - 1; ++t)
      if (t < ntiles) issue(t, t, page_of(t));
    page_next = page_of(C::NST - 1);
  }

  for (int t = 0; t < ntiles; ++t) {
    const int stage = t % C::NST;
    const uint32_t kbase = (FP8 && !C::REG8) ? sbase + C::WORK_OFF : sbase + stage * C::STAGE_BYTES;
    const uint32_t vbase = kbase + (C::REG8 ? C::K_LOAD : C::K_TILE);
    bool landed = mbar_wait(&full[stage], (phase >> stage) & 1u, p.wait_ns, nullptr);
    if (t == 0 && p.test_timeout) landed = mbar_wait(never, 0, kTestWaitNs, nullptr) && landed;
    phase ^= 1u << stage;
    const int nvalid = kend - (kstart + t * kTileKeys);
    if constexpr (C::REG8) {
      // V rows past the end may hold anything (NaN included): zero bytes there (K rows
      // there only feed masked scores)
      if (landed && nvalid < kTileKeys) {
        for (int idx = tid; idx < (kTileKeys - nvalid) * (DV / 16); idx += C::THREADS) {
          const int r = nvalid + idx / (DV / 16);
          *reinterpret_cast<uint4*>(smem + (vbase - sbase) + tile8_off(r, idx % (DV / 16))) = make_uint4(0, 0, 0, 0);
        }
      }
    } else if constexpr (FP8) {
      // widen the landed e4m3 tile pair into the bf16 work tiles (swizzled as the MMAs
      // read them). V rows past the end are written as zeros instead: they may hold
      // anything, NaN included (their P is 0, but 0 * NaN is NaN); K rows there only
      // feed masked scores. Every warp is done with the previous tile's work tiles (the
      // barrier at the end of the last iteration).
      if (landed) {
        const uint8_t* src = smem + stage * C::STAGE_BYTES;
        constexpr int KCH = DK / 16, VCH = DV / 16;  // 16-byte (16-value) chunks per row
        for (int idx = tid; idx < kTileKeys * (KCH + VCH); idx += C::THREADS) {
          const bool isv = idx >= kTileKeys * KCH;
          const int j = isv ? idx - kTileKeys * KCH : idx;
          const int ch = isv ? VCH : KCH;
          const int r = j / ch, u = j % ch;
          uint4 w0 = make_uint4(0, 0, 0, 0), w1 = make_uint4(0, 0, 0, 0);
          if (!isv || r < nvalid) {
            const uint4 b = *reinterpret_cast<const uint4*>(src + (isv ? C::K_LOAD + r * DV : r * DK) + u * 16);
            w0 = make_uint4(e4m3x2_to_bf16x2(b.x & 0xffffu), e4m3x2_to_bf16x2(b.x >> 16),
                            e4m3x2_to_bf16x2(b.y & 0xffffu), e4m3x2_to_bf16x2(b.y >> 16));
            w1 = make_uint4(e4m3x2_to_bf16x2(b.z & 0xffffu), e4m3x2_to_bf16x2(b.z >> 16),
                            e4m3x2_to_bf16x2(b.w & 0xffffu), e4m3x2_to_bf16x2(b.w >> 16));
          }
          uint8_t* dst = smem + C::WORK_OFF + (isv ? C::K_TILE : 0);
          *reinterpret_cast<uint4*>(dst + tile_off(r, 2 * u)) = w0;
          *reinterpret_cast<uint4*>(dst + tile_off(r, 2 * u + 1)) = w1;
        }
      }
    } else if (landed && nvalid < kTileKeys) {
      // V rows past the end of the segment may hold anything (NaN included): their P is
      // 0, but 0 * NaN is NaN in P V, so they are zeroed (K rows there only feed masked
      // scores)
      for (int idx = tid; idx < (kTileKeys - nvalid) * (DV / 8); idx += C::THREADS) {
        const int r = nvalid + idx / (DV / 8);
        *reinterpret_cast<uint4*>(smem + (vbase - sbase) + tile_off(r, idx % (DV / 8))) = make_uint4(0, 0, 0, 0);
      }
    }
    // tile t complete for everyone; every warp is done with tile t-1's stage
    if (__syncthreads_or(!landed)) {
      // A wait ran out (in some thread): record it, let the copies already requested
      // (tiles t .. t+NST-2) land before the CTA leaves their shared memory, and stop.
      if (tid == 0) {
        raise_error(p.err, kErrWaitTimeout);
        for (int j = 0; j < C::NST - 1 && t + j < ntiles; ++j) {
          const int st = (t + j) % C::NST;
          const uint32_t par = ((phase >> st) & 1u) ^ (j == 0 ? 1u : 0u);  // tile t's bit already moved on
          mbar_wait(&full[st], par, kTeardownNs, nullptr);
        }
      }
      __syncthreads();
      return false;
    }
    if (tid == 0 && t + C::NST - 1 < ntiles) {
      issue(t + C::NST - 1, (t + C::NST - 1) % C::NST, page_next);
      page_next = page_of(t + C::NST);
    }
    const int key_w = kstart + t * kTileKeys + slice * 16;  // first key of this warp's slice

    // S = Q K^T over the 16 keys of the slice (two n-tiles of 8 keys); for d >= 128 the
    // k-steps alternate between two accumulator sets, halving the dependent MMA chain.
    float sc[2][4];
    {
      constexpr int NACC = KS >= 8 ? 2 : 1;
      float sacc[NACC][2][4];
#pragma unroll
      for (int a = 0; a < NACC; ++a)
#pragma unroll
        for (int n = 0; n < 2; ++n) sacc[a][n][0] = sacc[a][n][1] = sacc[a][n][2] = sacc[a][n][3] = 0.f;
      if constexpr (C::REG8) {
        // byte tile: matrices (keys 0-7 | 8-15 of the slice) x (16-dim chunks 2kp | 2kp+1);
        // a thread's 32 bits are dimensions 4c .. 4c+3 of one key, widened to two f16 pairs
        const int kr = slice * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
        for (int kp = 0; kp < KS / 2; ++kp) {
          uint32_t r[4], lo[4], hi[4];
          ldmatrix_x4(kbase + tile8_off(kr, kp * 2 + (lane >> 4)), r[0], r[1], r[2], r[3]);
#pragma unroll
          for (int i = 0; i < 4; ++i) e4m3x4_to_f16x2x2(r[i], lo[i], hi[i]);
          mma_f16_16816(sacc[(2 * kp) % NACC][0], qa[2 * kp], lo[0], hi[0]);
          mma_f16_16816(sacc[(2 * kp) % NACC][1], qa[2 * kp], lo[1], hi[1]);
          mma_f16_16816(sacc[(2 * kp + 1) % NACC][0], qa[2 * kp + 1], lo[2], hi[2]);
          mma_f16_16816(sacc[(2 * kp + 1) % NACC][1], qa[2 * kp + 1], lo[3], hi[3]);
        }
      } else {
        const int kr = slice * 16 + (lane & 7) + ((lane >> 4) & 1) * 8;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          const int c = ks * 2 + ((lane >> 3) & 1);
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4(kbase + tile_off(kr, c), b0, b1, b2, b3);
          mma_bf16_16816(sacc[ks % NACC][0], qa[ks], b0, b1);
          mma_bf16_16816(sacc[ks % NACC][1], qa[ks], b2, b3);
        }
      }
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float v = sacc[0][n][e];
#pragma unroll
          for (int a = 1; a < NACC; ++a) v += sacc[a][n][e];
          sc[n][e] = v;
        }
    }

    // online softmax (exp2 domain); P packed as bf16 A fragments. The reference maximum
    // of a row moves only when the row's maximum grows by more than 2^8 (P values stay
    // below 256, exact enough in bf16 with fp32 sums), so the 2*NT-register rescale of the
    // output accumulator is skipped on almost every tile.
    uint32_t pa[4];
    float alpha2[2] = {1.f, 1.f};
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      float x[4];
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int key = key_w + n * 8 + (lane & 3) * 2 + e;
          x[n * 2 + e] = key < lim[h2] ? sc[n][h2 * 2 + e] * p.scale_log2 : -INFINITY;
        }
      float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      if (mx > m_run[h2] + kRescaleLog2) {
        alpha2[h2] = fast_exp2(m_run[h2] - mx);  // 0 while nothing was seen yet
        m_run[h2] = mx;
      }
      const float ref = m_run[h2] == -INFINITY ? 0.f : m_run[h2];
      float pv[4], ps = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        pv[e] = fast_exp2(x[e] - ref);  // masked keys -> 0
        ps += pv[e];
      }
      l_run[h2] = l_run[h2] * alpha2[h2] + ps;
      pa[h2 + 0] = C::REG8 ? pack_f16(pv[0], pv[1]) : pack_bf16(pv[0], pv[1]);  // keys 0-7 of the slice
      pa[h2 + 2] = C::REG8 ? pack_f16(pv[2], pv[3]) : pack_bf16(pv[2], pv[3]);  // keys 8-15
    }
    if (__any_sync(0xffffffffu, alpha2[0] != 1.f || alpha2[1] != 1.f)) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        o[nt][0] *= alpha2[0];
        o[nt][1] *= alpha2[0];
        o[nt][2] *= alpha2[1];
        o[nt][3] *= alpha2[1];
      }
    }

    // O += P V (V fragments through ldmatrix.trans)
    if constexpr (C::REG8) {
      // byte tile through ldmatrix.trans: a thread's 32 bits are two keys (2c, 2c+1) x two
      // dimensions (2p, 2p+1) of a 16-dim chunk; bytes 0/2 give the even dimension's key
      // pair, bytes 1/3 the odd one's, so each chunk feeds two n-tiles: even dimensions
      // (accumulator 2u) and odd dimensions (2u + 1); the merge below un-permutes them
      const int kr = slice * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
      for (int up = 0; up < DV / 32; ++up) {
        uint32_t r[4], ev[4], od[4];
        ldmatrix_x4_trans(vbase + tile8_off(kr, up * 2 + (lane >> 4)), r[0], r[1], r[2], r[3]);
        // bytes (0, 2, 1, 3): the even dimension's key pair low, the odd one's high
#pragma unroll
        for (int i = 0; i < 4; ++i) e4m3x4_to_f16x2x2(__byte_perm(r[i], 0, 0x3120), ev[i], od[i]);
        mma_f16_16816(o[4 * up + 0], pa, ev[0], ev[1]);
        mma_f16_16816(o[4 * up + 1], pa, od[0], od[1]);
        mma_f16_16816(o[4 * up + 2], pa, ev[2], ev[3]);
        mma_f16_16816(o[4 * up + 3], pa, od[2], od[3]);
      }
    } else {
      const int kr = slice * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
      for (int dp = 0; dp < DV / 16; ++dp) {
        const int c = dp * 2 + ((lane >> 4) & 1);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(vbase + tile_off(kr, c), b0, b1, b2, b3);
        mma_bf16_16816(o[2 * dp], pa, b0, b1);
        mma_bf16_16816(o[2 * dp + 1], pa, b2, b3);
      }
    }
    if constexpr (FP8 && !C::REG8) __syncthreads();  // the next tile is widened into the same work tiles
  }
  __syncthreads();  // every copy has been consumed; the merge buffer below reuses the stages

  // ---- merge the four key slices of each m-tile through shared memory
  float* red_o = reinterpret_cast<float*>(smem);  // [MT][kSlices][16][OSTR]
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    float l = l_run[h2];
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    if ((lane & 3) == 0) {
      const int r = (lane >> 2) + h2 * 8;
      s_m[mt][slice][r] = m_run[h2];
      s_l[mt][slice][r] = l;
    }
  }
  __syncthreads();
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    const int r = (lane >> 2) + h2 * 8;
    float M = s_m[mt][0][r];
#pragma unroll
    for (int w = 1; w < kSlices; ++w) M = fmaxf(M, s_m[mt][w][r]);
    const float f = (M == -INFINITY) ? 0.f : exp2f(m_run[h2] - M);
    if constexpr (C::REG8) {
      // accumulator 2u + parity, column n holds dimension 16u + 2n + parity
      float* dst = red_o + ((mt * kSlices + slice) * 16 + r) * C::OSTR + (lane & 3) * 4;
#pragma unroll
      for (int u = 0; u < DV / 16; ++u) {
        *reinterpret_cast<float2*>(dst + u * 16) = make_float2(o[2 * u][h2 * 2] * f, o[2 * u + 1][h2 * 2] * f);
        *reinterpret_cast<float2*>(dst + u * 16 + 2) =
            make_float2(o[2 * u][h2 * 2 + 1] * f, o[2 * u + 1][h2 * 2 + 1] * f);
      }
    } else {
      float* dst = red_o + ((mt * kSlices + slice) * 16 + r) * C::OSTR + (lane & 3) * 2;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        *reinterpret_cast<float2*>(dst + nt * 8) = make_float2(o[nt][h2 * 2] * f, o[nt][h2 * 2 + 1] * f);
    }
  }
  __syncthreads();

  // ---- final rows (one chunk) or fp32 partials
  for (int idx = tid; idx < 16 * MT * (DV / 4); idx += C::THREADS) {
    const int rr = idx / (DV / 4);  // row within the CTA
    const int c4 = (idx % (DV / 4)) * 4;
    const int m2 = rr / 16, r = rr % 16;
    const int rg = rb * MT * 16 + rr;
    if (rg >= p.R) continue;
    float M = s_m[m2][0][r];
#pragma unroll
    for (int w = 1; w < kSlices; ++w) M = fmaxf(M, s_m[m2][w][r]);
    float Lsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kSlices; ++w) {
      if (M != -INFINITY) Lsum += s_l[m2][w][r] * exp2f(s_m[m2][w][r] - M);
      const float* src = red_o + ((m2 * kSlices + w) * 16 + r) * C::OSTR + c4;
      const float2 a0 = *reinterpret_cast<const float2*>(src);
      const float2 a1 = *reinterpret_cast<const float2*>(src + 2);
      acc.x += a0.x;
      acc.y += a0.y;
      acc.z += a1.x;
      acc.w += a1.y;
    }
    const float inv = Lsum > 0.f ? p.v_scale / Lsum : 0.f;  // v_scale: 1 unless the cache is FP8
    acc.x *= inv;
    acc.y *= inv;
    acc.z *= inv;
    acc.w *= inv;
    const float lse = Lsum > 0.f ? (M + log2f(Lsum)) * kLn2 : -INFINITY;
    const int j = g * p.G + rg / p.s;
    const size_t rowflat = (size_t)(bi * p.hq + j) * p.s + (rg % p.s);
    if (out_mode == kSegFinal) {
      uint2 pk;
      pk.x = pack_bf16(acc.x, acc.y);
      pk.y = pack_bf16(acc.z, acc.w);
      *reinterpret_cast<uint2*>(p.out + rowflat * DV + c4) = pk;
      if (p.lse && c4 == 0) p.lse[rowflat] = lse;
    } else if (out_mode == kSegSplit) {
      *reinterpret_cast<float4*>(p.ws_o + (rowflat * p.nsplit + slot) * DV + c4) = acc;
      if (c4 == 0) p.ws_lse[rowflat * p.nsplit + slot] = lse;
    } else {
      const size_t rec_row = (size_t)slot * (16 * MT) + rr;
      *reinterpret_cast<float4*>(p.ws_o + rec_row * DV + c4) = acc;
      if (c4 == 0) p.ws_lse[rec_row] = lse;
    }
  }
  __syncthreads();  // the merge buffer aliases the pipeline of the next segment
  return true;
}

// CTA set-up shared by both kernels (touches only shared memory and kernel parameters):
// the stage barriers (full[0 .. NST-1]), one barrier that nothing ever signals
// (full[NST], waited on by the forced-timeout test) and the tensor-map prefetch. False (for every thread) when the
// dynamic shared memory is not 1024-byte aligned, which the 128-byte swizzle needs.
template <int NST>
__device__ __forceinline__ bool cta_setup(const GqaParams& p, const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                          uint64_t* full, uint8_t* smem) {
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) raise_error(p.err, kErrLaunch);
    return false;
  }
  if (threadIdx.x == 0) {
#pragma unroll
    for (int i = 0; i <= NST; ++i) mbar_init(&full[i], 1);
    fence_mbar_init();
    prefetch_tmap(tm_k);
    prefetch_tmap(tm_v);
  }
  __syncthreads();
  return true;
}

// One CTA per (sequence, KV head, context chunk, block of query rows).
template <int DK, int DV, int MT, bool FP8>
__global__ void __launch_bounds__(128 * MT)
    gqa_split_kernel(GqaParams p, const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
  using C = GqaCfg<DK, DV, MT, FP8>;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ float s_m[MT][kSlices][16];
  __shared__ float s_l[MT][kSlices][16];
  __shared__ uint64_t full[C::NST + 1];  // stage landed (TMA transaction count); + the never-signalled one
  if (!cta_setup<C::NST>(p, &tm_k, &tm_v, full, smem)) return;
  uint32_t phase = 0;  // parity of each stage's next completion
  pdl_wait();  // queries, cache and lengths may come from the previous kernel in the stream
  pdl_trigger();
  const int tid = threadIdx.x;
  const int rb = blockIdx.x % p.nrb;
  const int split = blockIdx.x / p.nrb;
  const int g = blockIdx.y;
  const int bi = blockIdx.z;
  const int L = p.seqlens[bi];
  const int kstart = split * p.chunk;
  if (kstart >= L) {  // chunk past the end: the combine skips it
    if (L <= 0 && p.nsplit == 1) {  // empty sequence without a combine pass: zero rows, LSE = -inf
      for (int idx = tid; idx < 16 * MT * (DV / 8); idx += C::THREADS) {
        const int rg = rb * MT * 16 + idx / (DV / 8);
        if (rg >= p.R) continue;
        const size_t rowflat = (size_t)(bi * p.hq + g * p.G + rg / p.s) * p.s + (rg % p.s);
        *reinterpret_cast<uint4*>(p.out + rowflat * DV + (idx % (DV / 8)) * 8) = make_uint4(0, 0, 0, 0);
        if (p.lse && idx % (DV / 8) == 0) p.lse[rowflat] = -INFINITY;
      }
    }
    return;
  }
  const int kend = min(L, kstart + p.chunk);
  gqa_segment<DK, DV, MT, FP8>(p, &tm_k, &tm_v, full, full + C::NST, phase, smem, s_m, s_l, bi, g, rb, L, kstart,
                               kend, p.nsplit == 1 ? kSegFinal : kSegSplit, split);
}

__device__ __forceinline__ long long tiles_of(int L) { return L > 0 ? (L + kTileKeys - 1) / kTileKeys : 0; }

// Balanced schedule. The work items (sequence, KV head, row block) are laid end to
// end in sequence-major order, each as its ceil(L/64) key tiles, and CTA c takes the
// tiles [c*W, (c+1)*W) with W = ceil(total / gridDim.x): every CTA gets the same
// number of tiles whatever the length mix, and a range may cut items anywhere. A
// piece that is a whole item is written as final rows; the pieces of a cut item go
// to partial records (record id = item index + CTA index, unique and increasing along
// the order) and the CTA holding the item's first tile stores {first record, count}
// in meta for the combine kernel. Computed from seqlens on the device, so the launch
// needs only an upper bound of the lengths.
template <int DK, int DV, int MT, bool FP8>
__global__ void __launch_bounds__(128 * MT)
    gqa_balanced_kernel(GqaParams p, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v) {
  using C = GqaCfg<DK, DV, MT, FP8>;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ float s_m[MT][kSlices][16];
  __shared__ float s_l[MT][kSlices][16];
  __shared__ uint64_t full[C::NST + 1];  // stage landed (TMA transaction count); + the never-signalled one
  constexpr int NW = C::THREADS / 32;
  __shared__ long long s_wsum[NW];  // inclusive prefix of the warps' tile counts
  // walk state, kept in shared memory so that nothing but constants stays live in
  // registers across the (register-bound) segment body
  __shared__ long long s_base, s_pos, s_end, s_w;
  __shared__ int s_seq;
  if (!cta_setup<C::NST>(p, &tm_k, &tm_v, full, smem)) return;
  uint32_t phase = 0;  // parity of each stage's next completion (runs on across segments)
  bool aborted = false;  // a tile wait ran out: the walk goes on, writing meta only
  pdl_wait();  // queries, cache and lengths may come from the previous kernel in the stream
  pdl_trigger();
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int ips = p.hkv * p.nrb;  // work items per sequence
  // tiles of each thread's block of sequences, and their exclusive prefix (block scan)
  const int per = (p.b + C::THREADS - 1) / C::THREADS;
  const int i0 = min(p.b, tid * per), i1 = min(p.b, i0 + per);
  long long mine = 0;
  for (int i = i0; i < i1; ++i) mine += tiles_of(p.seqlens[i]);
  long long incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) s_wsum[warp] = incl;
  if (tid == 0) {
    s_seq = p.b;
    s_base = 0;
  }
  __syncthreads();
  if (warp == 0) {
    long long w = lane < NW ? s_wsum[lane] : 0;
#pragma unroll
    for (int o = 1; o < NW; o <<= 1) {
      const long long n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    if (lane < NW) s_wsum[lane] = w;
  }
  __syncthreads();
  const long long excl = incl - mine + (warp > 0 ? s_wsum[warp - 1] : 0);
  const long long total = s_wsum[NW - 1] * ips;
  const long long W = (total + gridDim.x - 1) / gridDim.x;
  long long pos = (long long)blockIdx.x * W;
  const long long end = min(total, pos + W);
  if (pos >= end) return;
  {  // the sequence holding tile `pos`: found by the one thread whose block contains it
    long long b0 = excl * ips;
    if (pos >= b0 && pos < b0 + mine * ips) {
      for (int i = i0; i < i1; ++i) {
        const long long st = tiles_of(p.seqlens[i]) * ips;
        if (pos < b0 + st) {
          s_seq = i;
          s_base = b0;
          break;
        }
        b0 += st;
      }
    }
  }
  if (tid == 0) {
    s_pos = pos;
    s_end = end;
    s_w = W;
  }
  __syncthreads();
#pragma unroll 1
  while (true) {
    const long long pos = s_pos, end = s_end, W = s_w;
    int i = s_seq;
    long long base = s_base;  // first flattened tile of sequence i
    long long nt = 0;
    int L = 0;
    for (; i < p.b; ++i) {  // skip to the sequence holding tile pos (past ones, empty ones)
      L = p.seqlens[i];
      nt = tiles_of(L);
      if (pos < base + nt * ips) break;
      base += nt * ips;
    }
    if (pos >= end || i >= p.b) break;
    const long long off = pos - base;
    const int item_local = (int)(off / nt);
    const int t0 = (int)(off % nt);
    const int t1 = (int)min(nt, (long long)t0 + (end - pos));
    const int g = item_local / p.nrb;
    const int rb = item_local % p.nrb;
    const long long item = (long long)i * ips + item_local;
    const long long first = base + (long long)item_local * nt;  // flattened first tile of the item
    const int c0 = (int)(first / W);
    const int c1 = (int)((first + nt - 1) / W);
    if (t0 == 0 && tid == 0) {
      p.meta[2 * item] = (int)(item + c0);
      p.meta[2 * item + 1] = c1 - c0 + 1;
    }
    // After a time-out the remaining pieces are not computed, but every item whose first
    // tile lies in this CTA's range still gets its meta entry, so the combine reads only
    // records inside the workspace.
    if (!aborted)
      aborted = !gqa_segment<DK, DV, MT, FP8>(p, &tm_k, &tm_v, full, full + C::NST, phase, smem, s_m, s_l, i, g, rb, L,
                                         t0 * kTileKeys, min(L, t1 * kTileKeys), c0 == c1 ? kSegFinal : kSegRecord,
                                         (int)(item + blockIdx.x));
    else
      __syncthreads();
    // (both branches end with a barrier: every thread has read the state above)
    if (tid == 0) {
      s_pos = pos + (t1 - t0);
      s_seq = i;
      s_base = base;
    }
    __syncthreads();
  }
}

template <int DK, int DV, int MT, bool FP8 = false>
cudaError_t launch_gqa_dm(const GqaParams& p, int nsplit, int hkv, int b, int balanced_grid, cudaStream_t stream) {
  using C = GqaCfg<DK, DV, MT, FP8>;
  static std::atomic<unsigned long long> split_attr{0}, balanced_attr{0};
  if (cudaError_t e = ensure_smem_limit(gqa_split_kernel<DK, DV, MT, FP8>, C::SMEM, split_attr)) return e;
  if (cudaError_t e = ensure_smem_limit(gqa_balanced_kernel<DK, DV, MT, FP8>, C::SMEM, balanced_attr)) return e;
  // K and V as [tokens, KV heads, width] (contiguous: tokens = b x capacity; paged:
  // pages x 64). bf16: viewed as {64 values, tokens, width / 64 chunks, KV heads}
  // (strides: token hkv*width*2 B, chunk 128 B, head width*2 B), so that one box {64, 64
  // tokens, all chunks, 1 head} per tile lands chunk-major with 128-byte swizzled rows
  // (one request per tile instead of one per 64-dim chunk: 0.5-0.7 % faster on the
  // paged d = 256 shapes). FP8: byte boxes of one head's 64 tokens, as set out below.
  CUtensorMap tk, tv;
  {
    const uint64_t tokens = p.paged ? (uint64_t)p.num_pages * kTileKeys : (uint64_t)p.b * p.capacity;
    const cuuint64_t kdims[3] = {(cuuint64_t)DK, (cuuint64_t)p.hkv, (cuuint64_t)tokens};
    const cuuint64_t kstrides[2] = {(cuuint64_t)DK * C::CACHE_ELEM, (cuuint64_t)p.hkv * DK * C::CACHE_ELEM};
    const cuuint64_t vdims[3] = {(cuuint64_t)DV, (cuuint64_t)p.hkv, (cuuint64_t)tokens};
    const cuuint64_t vstrides[2] = {(cuuint64_t)DV * C::CACHE_ELEM, (cuuint64_t)p.hkv * DV * C::CACHE_ELEM};
    if (C::REG8) {  // bytes, [64 tokens x 128 bytes] boxes, 128-byte swizzle (ldmatrix reads them)
      const cuuint32_t box[3] = {128, 1, kTileKeys};
      if (!encode_tmap(&tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.k, 3, kdims, kstrides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
          !encode_tmap(&tv, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.v, 3, vdims, vstrides, box, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    } else if (FP8) {  // bytes, one box per tile, no swizzle (the widening pass reads rows linearly)
      const cuuint32_t kbox[3] = {(cuuint32_t)DK, 1, kTileKeys};
      const cuuint32_t vbox[3] = {(cuuint32_t)DV, 1, kTileKeys};
      if (!encode_tmap_u8(&tk, p.k, 3, kdims, kstrides, kbox) || !encode_tmap_u8(&tv, p.v, 3, vdims, vstrides, vbox))
        return cudaErrorInvalidValue;
    } else {
      const cuuint32_t kbox4[4] = {64, kTileKeys, (cuuint32_t)(DK / 64), 1};
      const cuuint32_t vbox4[4] = {64, kTileKeys, (cuuint32_t)(DV / 64), 1};
      const cuuint64_t kdims4[4] = {64, (cuuint64_t)tokens, (cuuint64_t)(DK / 64), (cuuint64_t)p.hkv};
      const cuuint64_t kstrides4[3] = {(cuuint64_t)p.hkv * DK * 2, 128, (cuuint64_t)DK * 2};
      const cuuint64_t vdims4[4] = {64, (cuuint64_t)tokens, (cuuint64_t)(DV / 64), (cuuint64_t)p.hkv};
      const cuuint64_t vstrides4[3] = {(cuuint64_t)p.hkv * DV * 2, 128, (cuuint64_t)DV * 2};
      if (!encode_tmap_bf16_sw128(&tk, p.k, 4, kdims4, kstrides4, kbox4) ||
          !encode_tmap_bf16_sw128(&tv, p.v, 4, vdims4, vstrides4, vbox4))
        return cudaErrorInvalidValue;
    }
  }
  // programmatic dependent launch: the CTAs may be scheduled while the previous kernel
  // finishes; they wait for it (pdl_wait) before reading anything
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = balanced_grid > 0 ? dim3(balanced_grid) : dim3(p.nrb * nsplit, hkv, b);
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = balanced_grid > 0 ? cudaLaunchKernelEx(&cfg, gqa_balanced_kernel<DK, DV, MT, FP8>, p, tk, tv)
                                          : cudaLaunchKernelEx(&cfg, gqa_split_kernel<DK, DV, MT, FP8>, p, tk, tv);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

// m-tiles per CTA: one for up to 16 query rows per KV head, else two
static int gqa_mt(int rows) { return rows <= 16 ? 1 : 2; }

int gqa_rows_per_cta(int rows) { return 16 * gqa_mt(rows); }

// Resident CTAs per SM of the balanced kernel (its grid is one wave of them).
template <int DK, int DV, int MT, bool FP8 = false>
static int balanced_occupancy() {
  using C = GqaCfg<DK, DV, MT, FP8>;
  // (the same GPU model on every device of a process is assumed for the cached value)
  static std::atomic<int> cached{0};
  static std::atomic<unsigned long long> attr{0};
  int n = cached.load(std::memory_order_relaxed);
  if (n == 0) {
    if (ensure_smem_limit(gqa_balanced_kernel<DK, DV, MT, FP8>, C::SMEM, attr) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gqa_balanced_kernel<DK, DV, MT, FP8>, C::THREADS, C::SMEM) !=
            cudaSuccess ||
        n <= 0)
      return 1;
    cached.store(n, std::memory_order_relaxed);
  }
  return n;
}

int gqa_balanced_ctas_per_sm(int dk, int dv, int rows, bool fp8) {
  const bool two = gqa_mt(rows) == 2;
  if (fp8) {
    switch (dk) {
      case 64: return two ? balanced_occupancy<64, 64, 2, true>() : balanced_occupancy<64, 64, 1, true>();
      case 128: return two ? balanced_occupancy<128, 128, 2, true>() : balanced_occupancy<128, 128, 1, true>();
      case 256: return two ? balanced_occupancy<256, 256, 2, true>() : balanced_occupancy<256, 256, 1, true>();
      default: return 1;
    }
  }
  if (dk == 192 && dv == 128) return two ? balanced_occupancy<192, 128, 2>() : balanced_occupancy<192, 128, 1>();
  if (dk != dv) return 1;
  switch (dk) {
    case 64: return two ? balanced_occupancy<64, 64, 2>() : balanced_occupancy<64, 64, 1>();
    case 128: return two ? balanced_occupancy<128, 128, 2>() : balanced_occupancy<128, 128, 1>();
    case 256: return two ? balanced_occupancy<256, 256, 2>() : balanced_occupancy<256, 256, 1>();
    default: return 1;
  }
}
int gqa_ctas_per_sm(int dk, int dv) {
  if (dk != dv) return 1;
  return dk <= 64 ? 3 : (dk <= 128 ? 2 : 1);
}
bool gqa_supported(int dk, int dv, bool fp8) {
  if (fp8) return dk == dv && (dk == 64 || dk == 128 || dk == 256);
  return (dk == dv && (dk == 64 || dk == 128 || dk == 256)) || (dk == 192 && dv == 128);
}

cudaError_t launch_gqa(const GqaLaunch& a, cudaStream_t stream) {
  GqaParams p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.k = static_cast<const __nv_bfloat16*>(a.k);
  p.v = static_cast<const __nv_bfloat16*>(a.v);
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
  const int mt = gqa_mt(p.R);
  p.nrb = (p.R + 16 * mt - 1) / (16 * mt);
  p.nsplit = a.nsplit;
  p.chunk = a.chunk;
  // FP8 cache: the key scale folds into the softmax scale, the value scale into the output
  p.scale_log2 = a.scale * (a.fp8 ? a.k_scale : 1.f) * kLog2e;
  p.v_scale = a.fp8 ? a.v_scale : 1.f;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.lse = a.lse;
  p.ws_o = a.ws_o;
  p.ws_lse = a.ws_lse;
  p.meta = a.meta;
  p.err = a.err;
  p.wait_ns = a.wait_ns;
  p.test_timeout = a.test_timeout;
#define DECATTN_GQA_CASE(DK, DV)                                                                     \
  if (!a.fp8 && a.dk == DK && a.dv == DV)                                                            \
    return mt == 1 ? launch_gqa_dm<DK, DV, 1>(p, a.nsplit, a.hkv, a.b, a.balanced_grid, stream)      \
                   : launch_gqa_dm<DK, DV, 2>(p, a.nsplit, a.hkv, a.b, a.balanced_grid, stream);
  DECATTN_GQA_CASE(64, 64)
  DECATTN_GQA_CASE(128, 128)
  DECATTN_GQA_CASE(256, 256)
#define DECATTN_GQA_FP8_CASE(D)                                                                      \
  if (a.dk == D && a.dv == D)                                                                        \
    return mt == 1 ? launch_gqa_dm<D, D, 1, true>(p, a.nsplit, a.hkv, a.b, a.balanced_grid, stream)  \
                   : launch_gqa_dm<D, D, 2, true>(p, a.nsplit, a.hkv, a.b, a.balanced_grid, stream);
  if (a.fp8) {
    DECATTN_GQA_FP8_CASE(64)
    DECATTN_GQA_FP8_CASE(128)
    DECATTN_GQA_FP8_CASE(256)
    return cudaErrorInvalidValue;
  }
  DECATTN_GQA_CASE(192, 128)
#undef DECATTN_GQA_CASE
#undef DECATTN_GQA_FP8_CASE
  return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------------------
// Split combine (log-sum-exp merge), shared by both attention forms.
// Row r of the output merges partials c < ceil(L / chunk) of its sequence:
//   lse = log sum_c exp(lse_c),  o = sum_c exp(lse_c - lse) o_c
// Partials whose rows saw no key carry lse_c = -inf and weigh nothing; a row
// with no partial (empty sequence) gets o = 0, lse = -inf.

// Combine geometry: D/8 threads per row (thread t owns columns 8t .. 8t+7), 256-thread
// blocks holding 256 / (D/8) rows, so that a launch is about one wave of small blocks.
template <int D>
struct MergeCfg {
  static constexpr int TPR = D / 8;
  static constexpr int ROWS = 256 / TPR;
};

// Partial element loads: 8 consecutive values (fp32 or bf16 partials).
__device__ __forceinline__ void load8(const float* p, float* v) {
  const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float* v) {
  const uint4 a = *reinterpret_cast<const uint4*>(p);
  v[0] = bf16_lo(a.x); v[1] = bf16_hi(a.x); v[2] = bf16_lo(a.y); v[3] = bf16_hi(a.y);
  v[4] = bf16_lo(a.z); v[5] = bf16_hi(a.z); v[6] = bf16_lo(a.w); v[7] = bf16_hi(a.w);
}

// The threads of one row merge its n partials: partial c has its D values at
// o0 + c * o_stride and its LSE at l0[c * l_stride]. Partials are taken U at a
// time with all their loads issued before any use (one memory round trip per
// group), merged with a running maximum; a partial with LSE = -inf saw no key and
// is skipped. (U = 2 where there are at most two partials: fewer registers, more
// blocks resident.) T is the partials' element type (fp32, or bf16 for the latent
// kernel's O / l partials).
template <int D, int U = 4, class T = float>
__device__ __forceinline__ void merge_row(const T* __restrict__ o0, size_t o_stride, const float* __restrict__ l0,
                                          size_t l_stride, int n, __nv_bfloat16* __restrict__ out_row,
                                          float* __restrict__ lse_out, int t) {
  float M = -INFINITY, wsum = 0.f;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  for (int c0 = 0; c0 < n; c0 += U) {
    float lv[U];
    float x[U][8];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      lv[u] = -INFINITY;
#pragma unroll
      for (int e = 0; e < 8; ++e) x[u][e] = 0.f;
      if (c0 + u < n) {
        lv[u] = l0[(size_t)(c0 + u) * l_stride];
        load8(o0 + (size_t)(c0 + u) * o_stride + 8 * t, x[u]);
      }
    }
    float mn = M;
#pragma unroll
    for (int u = 0; u < U; ++u) mn = fmaxf(mn, lv[u]);
    if (mn == -INFINITY) continue;
    const float f = expf(M - mn);  // 0 while nothing was merged yet
    wsum *= f;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] *= f;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (lv[u] == -INFINITY) continue;
      const float w = expf(lv[u] - mn);
      wsum += w;
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] += w * x[u][e];
    }
    M = mn;
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  uint4 pk;
  pk.x = pack_bf16(acc[0] * inv, acc[1] * inv);
  pk.y = pack_bf16(acc[2] * inv, acc[3] * inv);
  pk.z = pack_bf16(acc[4] * inv, acc[5] * inv);
  pk.w = pack_bf16(acc[6] * inv, acc[7] * inv);
  *reinterpret_cast<uint4*>(out_row + 8 * t) = pk;
  if (lse_out && t == 0) *lse_out = wsum > 0.f ? M + logf(wsum) : -INFINITY;
}

// Fixed chunks: row r merges partials c < ceil(L / chunk) of its sequence.
template <int D, int U, class T>
__global__ void __launch_bounds__(256) combine_kernel(const T* __restrict__ ws_o, const float* __restrict__ ws_lse,
                                                      const int32_t* __restrict__ seqlens, int rows,
                                                      int rows_per_seq, int nsplit, int chunk,
                                                      __nv_bfloat16* __restrict__ out, float* __restrict__ lse_out) {
  using M = MergeCfg<D>;
  pdl_wait();  // the partials come from the attention kernel just before
  pdl_trigger();
  const int row = blockIdx.x * M::ROWS + threadIdx.x / M::TPR;
  if (row >= rows) return;
  const int L = seqlens[row / rows_per_seq];
  const int nv = L > 0 ? min(nsplit, (L + chunk - 1) / chunk) : 0;
  merge_row<D, U, T>(ws_o + (size_t)row * nsplit * D, D, ws_lse + (size_t)row * nsplit, 1, nv, out + (size_t)row * D,
                     lse_out ? lse_out + row : nullptr, threadIdx.x % M::TPR);
}

// Combine for the balanced grouped-head schedule: row (bi, head j, token) belongs to
// work item (bi, KV head j / G, row block) whose meta entry gives its partial records;
// a whole item (one record) was written as final rows by its CTA, an empty sequence
// has no item and gets o = 0, LSE = -inf here.
template <int D>
__global__ void __launch_bounds__(256) combine_balanced_kernel(const float* __restrict__ ws_o,
                                                               const float* __restrict__ ws_lse,
                                                               const int* __restrict__ meta,
                                                               const int32_t* __restrict__ seqlens, int rows, int hq,
                                                               int s, int hkv, int G, int rpb, int nrb, long long records,
                                                               __nv_bfloat16* __restrict__ out,
                                                               float* __restrict__ lse_out) {
  using M = MergeCfg<D>;
  pdl_wait();  // the partials come from the attention kernel just before
  pdl_trigger();
  const int row = blockIdx.x * M::ROWS + threadIdx.x / M::TPR;
  if (row >= rows) return;
  const int bi = row / (hq * s);
  const int j = (row / s) % hq;
  const int r = (j % G) * s + row % s;  // row within the KV head's rows
  const long long item = ((long long)bi * hkv + j / G) * nrb + r / rpb;
  int first = 0, n = 0;
  if (seqlens[bi] > 0) {
    first = meta[2 * item];
    n = meta[2 * item + 1];
    if (n <= 1) return;  // written directly by its CTA
    // meta is written by the attention kernel for every item; the clamp only keeps a
    // corrupted entry from sending the loads outside the workspace
    if (first < 0 || first >= records) return;
    n = (int)min((long long)n, records - first);
  }
  const size_t rec_row = (size_t)first * rpb + r % rpb;
  merge_row<D>(ws_o + rec_row * D, (size_t)rpb * D, ws_lse + rec_row, (size_t)rpb, n, out + (size_t)row * D,
               lse_out ? lse_out + row : nullptr, threadIdx.x % M::TPR);
}

// The same merge for few rows with many partials each (the tensor-core kernel's balanced
// pieces give about SMs / items partials per row): one block per row. The partials are
// split over NG = 256 / (D / 8) groups of threads, each group merging its share with four
// partials' loads in flight per round; the groups' (maximum, weight sum, weighted row)
// are then combined through shared memory. A row of a whole item returns at once.
template <int D>
__global__ void __launch_bounds__(256) combine_wide_kernel(const float* __restrict__ ws_o,
                                                           const float* __restrict__ ws_lse,
                                                           const int* __restrict__ meta,
                                                           const int32_t* __restrict__ seqlens, int hq, int s, int hkv,
                                                           int G, int rpb, int nrb, long long records,
                                                           __nv_bfloat16* __restrict__ out,
                                                           float* __restrict__ lse_out) {
  constexpr int TPR = D / 8, NG = 256 / TPR;
  __shared__ float s_m[NG], s_w[NG];
  __shared__ __align__(16) float s_acc[NG][D];
  pdl_wait();  // the partials come from the attention kernel just before
  pdl_trigger();
  const int row = blockIdx.x;
  const int bi = row / (hq * s);
  const int j = (row / s) % hq;
  const int r = (j % G) * s + row % s;  // row within the KV head's rows
  const long long item = ((long long)bi * hkv + j / G) * nrb + r / rpb;
  int first = 0, n = 0;
  if (seqlens[bi] > 0) {
    first = meta[2 * item];
    n = meta[2 * item + 1];
    if (n <= 1) return;  // written directly by its CTA
    if (first < 0 || first >= records) return;  // only a corrupted entry: stay inside the workspace
    n = (int)min((long long)n, records - first);
  }
  const int g = threadIdx.x / TPR, t = threadIdx.x % TPR;
  const size_t rec_row = (size_t)first * rpb + r % rpb;
  const float* o0 = ws_o + rec_row * D + 8 * t;
  const float* l0 = ws_lse + rec_row;
  float M = -INFINITY, wsum = 0.f;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  for (int c0 = g; c0 < n; c0 += 4 * NG) {
    float lv[4];
    float x[4][8];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c = c0 + u * NG;
      lv[u] = -INFINITY;
#pragma unroll
      for (int e = 0; e < 8; ++e) x[u][e] = 0.f;
      if (c < n) {
        lv[u] = l0[(size_t)c * rpb];
        load8(o0 + (size_t)c * rpb * D, x[u]);
      }
    }
    float mn = M;
#pragma unroll
    for (int u = 0; u < 4; ++u) mn = fmaxf(mn, lv[u]);
    if (mn == -INFINITY) continue;
    const float f = expf(M - mn);  // 0 while nothing was merged yet
    wsum *= f;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] *= f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (lv[u] == -INFINITY) continue;
      const float w = expf(lv[u] - mn);
      wsum += w;
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] += w * x[u][e];
    }
    M = mn;
  }
  if (t == 0) {
    s_m[g] = M;
    s_w[g] = wsum;
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) s_acc[g][8 * t + e] = acc[e];
  __syncthreads();
  if (g != 0) return;
  float mx = -INFINITY;
#pragma unroll 4
  for (int gg = 0; gg < NG; ++gg) mx = fmaxf(mx, s_m[gg]);
  float W = 0.f;
  float a[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) a[e] = 0.f;
  if (mx != -INFINITY) {
    for (int gg = 0; gg < NG; ++gg) {
      if (s_m[gg] == -INFINITY) continue;
      const float f = expf(s_m[gg] - mx);
      W += f * s_w[gg];
#pragma unroll
      for (int e = 0; e < 8; ++e) a[e] += f * s_acc[gg][8 * t + e];
    }
  }
  const float inv = W > 0.f ? 1.f / W : 0.f;
  uint4 pk;
  pk.x = pack_bf16(a[0] * inv, a[1] * inv);
  pk.y = pack_bf16(a[2] * inv, a[3] * inv);
  pk.z = pack_bf16(a[4] * inv, a[5] * inv);
  pk.w = pack_bf16(a[6] * inv, a[7] * inv);
  *reinterpret_cast<uint4*>(out + (size_t)row * D + 8 * t) = pk;
  if (lse_out && t == 0) lse_out[row] = W > 0.f ? mx + logf(W) : -INFINITY;
}

// Combine of the latent MLA kernel's tail split: partial row rp belongs to unit
// tail_whole + rp / 128 (row tile mt of sequence bi), row rp % 128 of it; its k bf16
// partials cover chunks of `chunk` keys, of which ceil(L / chunk) saw keys.
template <int D>
__global__ void __launch_bounds__(256) combine_tail_kernel(const __nv_bfloat16* __restrict__ ws_o,
                                                           const float* __restrict__ ws_lse,
                                                           const int32_t* __restrict__ seqlens, int tail_rows,
                                                           int tail_whole, int mtiles, int rows_per_seq, int k, int chunk,
                                                           __nv_bfloat16* __restrict__ out, float* __restrict__ lse_out) {
  using M = MergeCfg<D>;
  pdl_wait();  // the partials come from the attention kernel just before
  pdl_trigger();
  const int rp = blockIdx.x * M::ROWS + threadIdx.x / M::TPR;
  if (rp >= tail_rows) return;
  const int u = tail_whole + rp / 128;
  const int bi = u / mtiles;
  const int rin = (u % mtiles) * 128 + rp % 128;  // row within the sequence
  if (rin >= rows_per_seq) return;
  const size_t row = (size_t)bi * rows_per_seq + rin;
  const int L = seqlens[bi];
  const int nv = L > 0 ? min(k, (L + chunk - 1) / chunk) : 0;
  merge_row<D, 2, __nv_bfloat16>(ws_o + (size_t)rp * k * D, D, ws_lse + (size_t)rp * k, 1, nv, out + row * D,
                                 lse_out ? lse_out + row : nullptr, threadIdx.x % M::TPR);
}

template <int D>
static int merge_blocks(int rows) {
  return (rows + MergeCfg<D>::ROWS - 1) / MergeCfg<D>::ROWS;
}

// The combine kernels are launched as programmatic dependents of the attention kernel
// before them: their blocks may be scheduled while its last CTAs run and wait in
// pdl_wait() for its results.
template <class K, class... A>
static cudaError_t launch_dependent(K kernel, int blocks, cudaStream_t stream, A... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <class T>
static cudaError_t launch_combine_t(const T* ws_o, const float* ws_lse, const int32_t* seqlens, int rows,
                                   int rows_per_seq, int nsplit, int chunk, int d, __nv_bfloat16* o, float* lse,
                                   cudaStream_t stream) {
#define DECATTN_COMBINE_CASE(D)                                                                                 \
  case D:                                                                                                       \
    return nsplit <= 2 ? launch_dependent(combine_kernel<D, 2, T>, merge_blocks<D>(rows), stream, ws_o, ws_lse,  \
                                          seqlens, rows, rows_per_seq, nsplit, chunk, o, lse)                    \
                       : launch_dependent(combine_kernel<D, 4, T>, merge_blocks<D>(rows), stream, ws_o, ws_lse,  \
                                          seqlens, rows, rows_per_seq, nsplit, chunk, o, lse);
  switch (d) {
    DECATTN_COMBINE_CASE(64)
    DECATTN_COMBINE_CASE(128)
    DECATTN_COMBINE_CASE(256)
    DECATTN_COMBINE_CASE(512)
    default: return cudaErrorInvalidValue;
  }
#undef DECATTN_COMBINE_CASE
}

cudaError_t launch_combine(const void* ws_o, bool bf16_partials, const float* ws_lse, const int32_t* seqlens, int rows,
                           int rows_per_seq, int nsplit, int chunk, int d, void* out, float* lse,
                           cudaStream_t stream) {
  auto* o = static_cast<__nv_bfloat16*>(out);
  const cudaError_t e =
      bf16_partials ? launch_combine_t(static_cast<const __nv_bfloat16*>(ws_o), ws_lse, seqlens, rows, rows_per_seq,
                                       nsplit, chunk, d, o, lse, stream)
                    : launch_combine_t(static_cast<const float*>(ws_o), ws_lse, seqlens, rows, rows_per_seq, nsplit,
                                       chunk, d, o, lse, stream);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_combine_tail(const void* ws_o, const float* ws_lse, const int32_t* seqlens, int tail_units,
                                int tail_whole, int mtiles, int rows_per_seq, int k, int chunk, int d, void* out,
                                float* lse, cudaStream_t stream) {
  const int tail_rows = tail_units * 128;
  const auto* o = static_cast<const __nv_bfloat16*>(ws_o);
  auto* dst = static_cast<__nv_bfloat16*>(out);
  cudaError_t e;
  switch (d) {
    case 512:
      e = launch_dependent(combine_tail_kernel<512>, merge_blocks<512>(tail_rows), stream, o, ws_lse, seqlens,
                           tail_rows, tail_whole, mtiles, rows_per_seq, k, chunk, dst, lse);
      break;
    case 64:
      e = launch_dependent(combine_tail_kernel<64>, merge_blocks<64>(tail_rows), stream, o, ws_lse, seqlens, tail_rows,
                           tail_whole, mtiles, rows_per_seq, k, chunk, dst, lse);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_combine_balanced(const float* ws_o, const float* ws_lse, const int* meta, const int32_t* seqlens,
                                    int b, int hq, int s, int hkv, int d, int rpb, long long records, void* out,
                                    float* lse, cudaStream_t stream) {
  const int rows_kv = (hq / hkv) * s;
  const int nrb = (rows_kv + rpb - 1) / rpb;
  const int rows = b * hq * s;
  auto* o = static_cast<__nv_bfloat16*>(out);
  const int G = hq / hkv;
  // few rows: one block per row, its partials merged by groups of threads in parallel
  const bool wide = rows <= 4096;
#define DECATTN_COMBINE_CASE(D)                                                                                  \
  case D:                                                                                                        \
    if (cudaError_t e = wide ? launch_dependent(combine_wide_kernel<D>, rows, stream, ws_o, ws_lse, meta, seqlens,  \
                                                hq, s, hkv, G, rpb, nrb, records, o, lse)                         \
                             : launch_dependent(combine_balanced_kernel<D>, merge_blocks<D>(rows), stream, ws_o,  \
                                                ws_lse, meta, seqlens, rows, hq, s, hkv, G, rpb, nrb, records, o, \
                                                lse))                                                             \
      return e;                                                                                                  \
    break;
  switch (d) {
    DECATTN_COMBINE_CASE(64)
    DECATTN_COMBINE_CASE(128)
    DECATTN_COMBINE_CASE(256)
    default: return cudaErrorInvalidValue;
  }
#undef DECATTN_COMBINE_CASE
  return cudaGetLastError();
}

}  // namespace decattn
