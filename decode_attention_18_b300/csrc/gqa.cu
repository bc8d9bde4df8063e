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
//  * K/V tiles of 64 keys stream through a 3-4 stage cp.async pipeline with
//    16-byte (128-bit) coalesced loads into XOR-swizzled shared memory.
//  * 4 warps per 16-row m-tile (MT m-tiles, 128*MT threads); each warp owns 16
//    keys of a tile: S = Q K^T and O += P V run on mma.sync m16n8k16 (bf16 in,
//    fp32 accumulate); the score fragment is reused in registers as the A
//    operand of P V.
//  * Online softmax per warp with quad shuffles (exp2 domain); the four key
//    slices of an m-tile are merged through shared memory at the end.
//  * Output: with one chunk, bf16 rows and the LSE directly; otherwise fp32
//    (O, LSE) partials for the combine kernel.
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
  unsigned* err;
};

constexpr int kTileKeys = 64;
constexpr int kSlices = 4;  // warps (key slices of 16) per m-tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.f;  // move a row's reference maximum only past 2^8

template <int D, int MT_>
struct GqaCfg {
  static constexpr int MT = MT_;  // 16-row m-tiles per CTA
  static constexpr int THREADS = 128 * MT;
  static constexpr int NST = D <= 64 ? 4 : 3;  // pipeline stages
  static constexpr int ROW_BYTES = D * 2;
  static constexpr int TILE_BYTES = kTileKeys * ROW_BYTES;  // one K (or V) tile
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int PIPE_BYTES = NST * STAGE_BYTES;
  static constexpr int OSTR = D + 2;  // padded fp32 row stride of the merge buffer
  static constexpr int RED_BYTES = kSlices * 16 * MT * OSTR * 4;
  static constexpr int SMEM = PIPE_BYTES > RED_BYTES ? PIPE_BYTES : RED_BYTES;
  static constexpr int CHUNKS = D / 8;  // 16-byte chunks per row
  static constexpr int LOADS = kTileKeys * CHUNKS / THREADS;
  static_assert(kTileKeys * CHUNKS % THREADS == 0, "tile load split");
};

__device__ __forceinline__ uint32_t swz(int row, int chunk) { return (uint32_t)(chunk ^ (row & 7)); }

template <int D, int MT>
__global__ void __launch_bounds__(128 * MT) gqa_split_kernel(GqaParams p) {
  using C = GqaCfg<D, MT>;
  constexpr int NT = D / 8;   // n-tiles of the output
  constexpr int KS = D / 16;  // k-steps of QK^T
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ float s_m[MT][kSlices][16];
  __shared__ float s_l[MT][kSlices][16];

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int mt = warp / kSlices;     // m-tile of this warp
  const int slice = warp % kSlices;  // 16-key slice of each tile
  const int rb = blockIdx.x % p.nrb;
  const int split = blockIdx.x / p.nrb;
  const int g = blockIdx.y;
  const int bi = blockIdx.z;

  const int L = p.seqlens[bi];
  const int kstart = split * p.chunk;
  if (kstart >= L) {  // chunk past the end: the combine skips it
    if (L <= 0 && p.nsplit == 1) {  // empty sequence without a combine pass: zero rows, LSE = -inf
      for (int idx = tid; idx < 16 * MT * (D / 8); idx += C::THREADS) {
        const int rg = rb * MT * 16 + idx / (D / 8);
        if (rg >= p.R) continue;
        const size_t rowflat = (size_t)(bi * p.hq + g * p.G + rg / p.s) * p.s + (rg % p.s);
        *reinterpret_cast<uint4*>(p.out + rowflat * D + (idx % (D / 8)) * 8) = make_uint4(0, 0, 0, 0);
        if (p.lse && idx % (D / 8) == 0) p.lse[rowflat] = -INFINITY;
      }
    }
    return;
  }
  const int kend = min(L, kstart + p.chunk);
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
      const int col = ks * 16 + (lane & 3) * 2 + (e >> 1) * 8;
      uint32_t val = 0;
      if (r < p.R) {
        const int j = g * p.G + r / p.s;
        const size_t off = ((size_t)(bi * p.hq + j) * p.s + (r % p.s)) * D + col;
        val = __ldg(reinterpret_cast<const unsigned int*>(p.q + off));
      }
      qa[ks][e] = val;
    }
  }

  // ---- K/V tile loader (all threads; zero-fill past the chunk end). For a paged cache
  // the tile's page index comes from page_of(); it is fetched one iteration ahead so that
  // the block-table read never sits in front of the copies.
  const uint32_t sbase = smem_u32(smem);
  auto page_of = [&](int t) -> int {
    const int key0 = kstart + t * kTileKeys;
    if (!p.paged || t >= ntiles) return 0;
    return __ldg(p.block_table + (size_t)bi * p.max_pages + key0 / kTileKeys);
  };
  // this thread's 16-byte chunks of a tile: row, shared-memory offset, element offset in the cache
  // (the element offset fits 32 bits: row < 64, hkv <= 65535, d <= 256)
  uint32_t ld_soff[C::LOADS];
  uint32_t ld_goff[C::LOADS];
#pragma unroll
  for (int n = 0; n < C::LOADS; ++n) {
    const int idx = tid + n * C::THREADS;
    const int kr = idx / C::CHUNKS;
    const int c = idx % C::CHUNKS;
    ld_soff[n] = kr * C::ROW_BYTES + swz(kr, c) * 16;
    ld_goff[n] = (uint32_t)(kr * p.hkv * D + c * 8);
  }
  auto load_tile = [&](int t, int stage, int page) {
    const int key0 = kstart + t * kTileKeys;
    long long rowbase;  // cache-tensor row of the tile's first token
    bool page_ok = true;
    if (p.paged) {
      if (page < 0 || page >= p.num_pages) {
        page_ok = false;
        if (tid == 0) raise_error(p.err, kErrBadPage);
      }
      rowbase = (long long)page * kTileKeys;
    } else {
      rowbase = (long long)bi * p.capacity + key0;
    }
    const uint32_t kdst = sbase + stage * C::STAGE_BYTES;
    const uint32_t vdst = kdst + C::TILE_BYTES;
    const __nv_bfloat16* kt = p.k + ((size_t)rowbase * p.hkv + g) * D;
    const __nv_bfloat16* vt = p.v + ((size_t)rowbase * p.hkv + g) * D;
    const int nvalid = page_ok ? kend - key0 : 0;  // keys of the tile inside the chunk
#pragma unroll
    for (int n = 0; n < C::LOADS; ++n) {
      const int kr = (tid + n * C::THREADS) / C::CHUNKS;
      const bool valid = kr < nvalid;
      const uint32_t goff = valid ? ld_goff[n] : 0u;
      cp_async_16(kdst + ld_soff[n], kt + goff, valid ? 16u : 0u);
      cp_async_16(vdst + ld_soff[n], vt + goff, valid ? 16u : 0u);
    }
  };

  // ---- online-softmax state and output accumulator (rows lane/4 and lane/4 + 8)
  float o[NT][4];
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;

#pragma unroll
  for (int t = 0; t < C::NST - 1; ++t) {
    if (t < ntiles) load_tile(t, t, page_of(t));
    cp_async_commit();
  }
  int page_next = page_of(C::NST - 1);  // page of the next tile to load

  for (int t = 0; t < ntiles; ++t) {
    cp_async_wait<C::NST - 2>();
    __syncthreads();
    {
      const int tn = t + C::NST - 1;
      const int page = page_next;
      page_next = page_of(tn + 1);
      if (tn < ntiles) load_tile(tn, tn % C::NST, page);
      cp_async_commit();
    }
    const int stage = t % C::NST;
    const uint32_t kbase = sbase + stage * C::STAGE_BYTES;
    const uint32_t vbase = kbase + C::TILE_BYTES;
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
      const int kr = slice * 16 + (lane & 7) + ((lane >> 4) & 1) * 8;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const int c = ks * 2 + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(kbase + kr * C::ROW_BYTES + swz(kr, c) * 16, b0, b1, b2, b3);
        mma_bf16_16816(sacc[ks % NACC][0], qa[ks], b0, b1);
        mma_bf16_16816(sacc[ks % NACC][1], qa[ks], b2, b3);
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
      pa[h2 + 0] = pack_bf16(pv[0], pv[1]);  // keys 0-7 of the slice
      pa[h2 + 2] = pack_bf16(pv[2], pv[3]);  // keys 8-15
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
    {
      const int kr = slice * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        const int c = dp * 2 + ((lane >> 4) & 1);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(vbase + kr * C::ROW_BYTES + swz(kr, c) * 16, b0, b1, b2, b3);
        mma_bf16_16816(o[2 * dp], pa, b0, b1);
        mma_bf16_16816(o[2 * dp + 1], pa, b2, b3);
      }
    }
  }
  cp_async_wait<0>();
  __syncthreads();

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
    float* dst = red_o + ((mt * kSlices + slice) * 16 + r) * C::OSTR + (lane & 3) * 2;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
      *reinterpret_cast<float2*>(dst + nt * 8) = make_float2(o[nt][h2 * 2] * f, o[nt][h2 * 2 + 1] * f);
  }
  __syncthreads();

  // ---- final rows (one chunk) or fp32 partials
  for (int idx = tid; idx < 16 * MT * (D / 4); idx += C::THREADS) {
    const int rr = idx / (D / 4);  // row within the CTA
    const int c4 = (idx % (D / 4)) * 4;
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
    const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
    acc.x *= inv;
    acc.y *= inv;
    acc.z *= inv;
    acc.w *= inv;
    const float lse = Lsum > 0.f ? (M + log2f(Lsum)) * kLn2 : -INFINITY;
    const int j = g * p.G + rg / p.s;
    const size_t rowflat = (size_t)(bi * p.hq + j) * p.s + (rg % p.s);
    if (p.nsplit == 1) {
      uint2 pk;
      pk.x = pack_bf16(acc.x, acc.y);
      pk.y = pack_bf16(acc.z, acc.w);
      *reinterpret_cast<uint2*>(p.out + rowflat * D + c4) = pk;
      if (p.lse && c4 == 0) p.lse[rowflat] = lse;
    } else {
      *reinterpret_cast<float4*>(p.ws_o + (rowflat * p.nsplit + split) * D + c4) = acc;
      if (c4 == 0) p.ws_lse[rowflat * p.nsplit + split] = lse;
    }
  }
}

template <int D, int MT>
cudaError_t launch_gqa_dm(const GqaParams& p, int nsplit, int hkv, int b, cudaStream_t stream) {
  using C = GqaCfg<D, MT>;
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e =
        cudaFuncSetAttribute(gqa_split_kernel<D, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  dim3 grid(p.nrb * nsplit, hkv, b);
  gqa_split_kernel<D, MT><<<grid, C::THREADS, C::SMEM, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

// m-tiles per CTA: one for up to 16 query rows per KV head, else two
static int gqa_mt(int rows) { return rows <= 16 ? 1 : 2; }

int gqa_rows_per_cta(int rows) { return 16 * gqa_mt(rows); }
int gqa_ctas_per_sm(int d) { return d <= 64 ? 3 : (d <= 128 ? 2 : 1); }

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
  p.scale_log2 = a.scale * kLog2e;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.lse = a.lse;
  p.ws_o = a.ws_o;
  p.ws_lse = a.ws_lse;
  p.err = a.err;
#define DECATTN_GQA_CASE(D)                                                        \
  case D:                                                                          \
    return mt == 1 ? launch_gqa_dm<D, 1>(p, a.nsplit, a.hkv, a.b, stream)          \
                   : launch_gqa_dm<D, 2>(p, a.nsplit, a.hkv, a.b, stream);
  switch (a.d) {
    DECATTN_GQA_CASE(64)
    DECATTN_GQA_CASE(128)
    DECATTN_GQA_CASE(256)
    default:
      return cudaErrorInvalidValue;
  }
#undef DECATTN_GQA_CASE
}

// ---------------------------------------------------------------------------
// Split combine (log-sum-exp merge), shared by both attention forms.
// Row r of the output merges partials c < ceil(L / chunk) of its sequence:
//   lse = log sum_c exp(lse_c),  o = sum_c exp(lse_c - lse) o_c
// Partials whose rows saw no key carry lse_c = -inf and weigh nothing; a row
// with no partial (empty sequence) gets o = 0, lse = -inf. One warp per row.

template <int D>
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ ws_o,
                                                      const float* __restrict__ ws_lse,
                                                      const int32_t* __restrict__ seqlens, int rows,
                                                      int rows_per_seq, int nsplit, int chunk,
                                                      __nv_bfloat16* __restrict__ out, float* __restrict__ lse_out) {
  constexpr int V = D / 32;  // floats per lane
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= rows) return;
  const int bi = warp / rows_per_seq;
  const int L = seqlens[bi];
  const int nv = min(nsplit, (L + chunk - 1) / chunk);
  const float* lrow = ws_lse + (size_t)warp * nsplit;
  float M = -INFINITY;
  for (int c = lane; c < nv; c += 32) M = fmaxf(M, lrow[c]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  constexpr int VEC = D >= 128 ? 4 : 2;  // floats per vector access
  float acc[V];
#pragma unroll
  for (int e = 0; e < V; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  if (M != -INFINITY) {
    for (int c = 0; c < nv; ++c) {
      const float w = expf(lrow[c] - M);
      wsum += w;
      if (w == 0.f) continue;
      const float* src = ws_o + ((size_t)warp * nsplit + c) * D + lane * VEC;
#pragma unroll
      for (int e = 0; e < V; e += VEC) {
        if constexpr (VEC == 4) {
          const float4 x = *reinterpret_cast<const float4*>(src + e * 32);
          acc[e + 0] += w * x.x;
          acc[e + 1] += w * x.y;
          acc[e + 2] += w * x.z;
          acc[e + 3] += w * x.w;
        } else {
          const float2 x = *reinterpret_cast<const float2*>(src + e * 32);
          acc[e + 0] += w * x.x;
          acc[e + 1] += w * x.y;
        }
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  __nv_bfloat16* dst = out + (size_t)warp * D + lane * VEC;
#pragma unroll
  for (int e = 0; e < V; e += VEC) {
    if constexpr (VEC == 4) {
      uint2 pk;
      pk.x = pack_bf16(acc[e + 0] * inv, acc[e + 1] * inv);
      pk.y = pack_bf16(acc[e + 2] * inv, acc[e + 3] * inv);
      *reinterpret_cast<uint2*>(dst + e * 32) = pk;
    } else {
      *reinterpret_cast<uint32_t*>(dst + e * 32) = pack_bf16(acc[e + 0] * inv, acc[e + 1] * inv);
    }
  }
  if (lse_out && lane == 0) lse_out[warp] = wsum > 0.f ? M + logf(wsum) : -INFINITY;
}

cudaError_t launch_combine(const float* ws_o, const float* ws_lse, const int32_t* seqlens, int rows,
                           int rows_per_seq, int nsplit, int chunk, int d, void* out, float* lse,
                           cudaStream_t stream) {
  const int threads = 256;
  const int blocks = (rows * 32 + threads - 1) / threads;
  auto* o = static_cast<__nv_bfloat16*>(out);
  switch (d) {
    case 64: combine_kernel<64><<<blocks, threads, 0, stream>>>(ws_o, ws_lse, seqlens, rows, rows_per_seq, nsplit, chunk, o, lse); break;
    case 128: combine_kernel<128><<<blocks, threads, 0, stream>>>(ws_o, ws_lse, seqlens, rows, rows_per_seq, nsplit, chunk, o, lse); break;
    case 256: combine_kernel<256><<<blocks, threads, 0, stream>>>(ws_o, ws_lse, seqlens, rows, rows_per_seq, nsplit, chunk, o, lse); break;
    case 512: combine_kernel<512><<<blocks, threads, 0, stream>>>(ws_o, ws_lse, seqlens, rows, rows_per_seq, nsplit, chunk, o, lse); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace decattn
