// Per-head projection GEMMs of the absorbed MLA pipeline (sm_103a).
//
// "Mla Analysis" skill page, "Absorption Trick (FlashMLA)": the score line
// folds the key up-projection into the query (Qz = q_nope W_uk, one GEMM per
// head) and the value line leaves the latent output to be decompressed by a
// separate kernel (O = O_lat W_uv). Both are batched per-head GEMMs
//   C[b, j, r, :] = scale * A[b, j, r, :] @ W[j]      (W[j] is kin x nout)
// with M = b*s rows per head. At decode sizes M is small (32 rows for 32
// sequences of one token) and the kernel is bound by reading W (h*kin*nout
// bf16, 16.8 MB for h=128, d=128, k=512), so it streams W once and runs
// mma.sync m16n8k16 (bf16, fp32 accumulate) on it. W arrives by TMA: one
// thread requests each k-stage as a single box of [64 k x BN n] (a 3-D view of W
// in 64-column chunks, 128-byte swizzle) on the stage's mbarrier. At decode sizes
// the CTA's whole weight slab fits in its stages, so every stage is requested at
// once, before the programmatic-launch wait (W is not an output of the previous
// kernel): one DRAM round trip per CTA, in as few and as large boxes as the
// swizzle allows. Issuing W as 16-byte cp.async copies instead costs one instruction per
// 16 bytes (thousands per CTA), which bounds the stream well below HBM speed.
// The activation rows (a few KB per CTA) still come by cp.async.
#include <cstring>

#include "common.cuh"
#include "internal.h"

namespace decattn {

namespace {

constexpr int BK = 64;

struct ProjParams {
  unsigned* err;
  unsigned long long wait_ns;
  const __nv_bfloat16* a;
  const __nv_bfloat16* w;
  __nv_bfloat16* c;
  const int32_t* seqlens;
  int b, s, h, kin, nout, M;
  float scale;
};

__device__ __forceinline__ uint32_t swz(int row, int chunk) { return (uint32_t)(chunk ^ (row & 7)); }

// One CTA: BM rows of one head x BN output columns, 4 warps laid out (BM/32) x (4/(BM/32)),
// each warp 32 rows x WN columns; NST k-stages of BK in flight. TMA_W: the W tile of a stage
// is BN/64 TMA boxes of [64 k x 64 n] (box-major, 128-byte swizzle); otherwise (narrow
// outputs) 16-byte cp.async copies with the same swizzle over BN*2-byte rows.
// Stage t holds k-tile t (t < NST) and then every NST-th one after it; all NST stages
// are requested before the first is consumed. SLAB (TMA_W, every k-tile fits its stage at
// once): the W stages are one slab [BN/64 chunks][NST*64 k][64 n] requested as boxes of
// up to 256 k-rows (one box per CTA at BN = 128, two at BN = 64 and 512 rows), since the
// TMA engine serves about one box per few hundred cycles per SM whatever its size.
template <int BM, int BN, int NST, bool TMA_W, bool SLAB>
__global__ void __launch_bounds__(128) proj_kernel(const __grid_constant__ CUtensorMap tm_w, ProjParams p) {
  constexpr int WMW = BM / 32;               // warps along M
  constexpr int WNW = 4 / WMW;               // warps along N
  constexpr int WN = BN / WNW;               // columns per warp
  constexpr int NTW = WN / 8;                // n-tiles per warp
  constexpr int A_BYTES = BM * BK * 2;       // [BM rows][64 k], rows of 128 B
  constexpr int B_ROW = BN * 2;              // bytes per k row of the W tile
  constexpr int B_BYTES = BK * B_ROW;        // [64 k][BN n]
  constexpr int STAGE = A_BYTES + B_BYTES;
  // slab boxes: KB k-rows each, NBOX of them
  constexpr int KB = NST * BK < 256 ? NST * BK : 256;
  constexpr int NBOX = (NST * BK + KB - 1) / KB;
  static_assert(NTW % 2 == 0 && (BM * 8) % 128 == 0 && (BK * (BN / 8)) % 128 == 0, "tile shape");
  static_assert(!TMA_W || (BN % 64 == 0 && A_BYTES % 1024 == 0 && STAGE % 1024 == 0), "TMA tile shape");
  static_assert(!SLAB || (TMA_W && (BN == 64 || NBOX == 1) && (NST * BK) % KB == 0), "slab boxes");
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ uint64_t wbar[NST];  // stage's (SLAB: box's) W landed (TMA)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wm = warp / WNW, wn = warp % WNW;
  const int n0 = blockIdx.x * BN;
  const int m0 = blockIdx.y * BM;
  const int j = blockIdx.z;
  const int kiters = (p.kin + BK - 1) / BK;
  const uint32_t sbase = smem_u32(smem);

  auto a_row_ptr = [&](int m) -> const __nv_bfloat16* {
    const int bi = m / p.s, i = m % p.s;
    return p.a + ((size_t)(bi * p.h + j) * p.s + i) * p.kin;
  };

  // SLAB: A stages [NST][A_BYTES], then the W slab; else stage t = A tile then W tile
  auto a_base = [&](int stage) -> uint32_t { return SLAB ? sbase + stage * A_BYTES : sbase + stage * STAGE; };
  auto load_a = [&](int kt, int stage) {
    const uint32_t adst = a_base(stage);
#pragma unroll
    for (int n = 0; n < (BM * 8) / 128; ++n) {
      const int idx = tid + n * 128;
      const int r = idx >> 3, c = idx & 7;
      const int m = m0 + r;
      const bool ok = m < p.M && kt * BK + c * 8 < p.kin;
      const __nv_bfloat16* src = ok ? a_row_ptr(m) + kt * BK + c * 8 : p.a;
      cp_async_16(adst + r * 128 + swz(r, c) * 16, src, ok ? 16u : 0u);
    }
  };
  // shared-memory offset of 16-byte chunk c (8 columns) of k-row r of a stage's W tile
  auto w_off = [&](int r, int c) -> uint32_t {
    if constexpr (SLAB) return (uint32_t)((c >> 3) * (NST * BK * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
    else if constexpr (TMA_W) return (uint32_t)((c >> 3) * (BK * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
    else return (uint32_t)(r * B_ROW + swz(r, c) * 16);
  };
  uint32_t wphase = 0;  // parity of each stage's next W completion (TMA_W)
  auto load_w = [&](int kt, int stage) {
    const uint32_t bdst = sbase + stage * STAGE + A_BYTES;
    if constexpr (SLAB) {
      (void)bdst;
      if (tid == 0 && kt * BK % KB == 0) {  // the box that starts at this k-tile
        const int bx = kt * BK / KB;
        mbar_expect_tx(&wbar[bx], KB * BN * 2);
        tma_load_3d(sbase + NST * A_BYTES + bx * KB * 128, &tm_w, 0, j * p.kin + kt * BK, n0 / 64, &wbar[bx]);
      }
      return;
    } else if constexpr (TMA_W) {
      if (tid == 0) {
        mbar_expect_tx(&wbar[stage], B_BYTES);
        tma_load_3d(bdst, &tm_w, 0, j * p.kin + kt * BK, n0 / 64, &wbar[stage]);
      }
      return;
    }
    const __nv_bfloat16* wbase = p.w + (size_t)j * p.kin * p.nout;
#pragma unroll
    for (int n = 0; n < (BK * (BN / 8)) / 128; ++n) {
      const int idx = tid + n * 128;
      const int r = idx / (BN / 8), c = idx % (BN / 8);
      const int kr = kt * BK + r, col = n0 + c * 8;
      const bool ok = kr < p.kin && col < p.nout;
      const __nv_bfloat16* src = ok ? wbase + (size_t)kr * p.nout + col : p.w;
      cp_async_16(bdst + r * B_ROW + swz(r, c) * 16, src, ok ? 16u : 0u);
    }
  };

  float acc[2][NTW][4];
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int ni = 0; ni < NTW; ++ni) acc[mi][ni][0] = acc[mi][ni][1] = acc[mi][ni][2] = acc[mi][ni][3] = 0.f;

  if constexpr (TMA_W) {
    if (smem_u32(smem) & 1023u) {  // the 128-byte swizzle needs 1024-byte aligned stages
      if (tid == 0) raise_error(p.err, kErrLaunch);
      return;
    }
    if (tid == 0) {
#pragma unroll
      for (int i = 0; i < (SLAB ? NBOX : NST); ++i) mbar_init(&wbar[i], 1);
      fence_mbar_init();
      prefetch_tmap(&tm_w);
    }
    __syncthreads();
  }
  // The weight does not come from the previous kernel in the stream: its stages are
  // requested before pdl_wait, so they load while that kernel finishes. (With cp.async
  // they join the first commit group, whose completion is awaited before stage 0 is
  // used; with TMA each stage has its barrier.) Commit group t carries k-tile t.
#pragma unroll
  for (int t = 0; t < NST; ++t)
    if (t < kiters) load_w(t, t);
  pdl_wait();  // the activations (and lengths) are the previous kernel's results
  pdl_trigger();
#pragma unroll
  for (int t = 0; t < NST; ++t) {
    if (t < kiters) load_a(t, t);
    cp_async_commit();
  }
  bool w_ok = true;
  for (int kt = 0; kt < kiters; ++kt) {
    // groups 0 .. kt+1 complete: k-tile t < NST is group t, a later one is group t + 1
    // (the iteration that refills it commits after the empty commit of iteration 0)
    cp_async_wait<NST - 2>();
    if constexpr (SLAB) {
      if (kt * BK % KB == 0) {  // the first k-tile of a box: wait for the box
        const int bx = kt * BK / KB;
        if (!mbar_wait(&wbar[bx], 0, p.wait_ns, nullptr)) {
          w_ok = false;  // recorded below; the box is waited for before the CTA leaves
          mbar_wait(&wbar[bx], 0, 1000000000ull, nullptr);
        }
      }
    } else if constexpr (TMA_W) {
      const int stage = kt % NST;
      if (!mbar_wait(&wbar[stage], (wphase >> stage) & 1u, p.wait_ns, nullptr)) {
        w_ok = false;  // recorded below; the stage's copy is waited for before the CTA leaves
        mbar_wait(&wbar[stage], (wphase >> stage) & 1u, 1000000000ull, nullptr);
      }
      wphase ^= 1u << stage;
    }
    __syncthreads();  // every warp is done with stage (kt - 1) % NST
    if (kt >= 1 && kt - 1 + NST < kiters) {
      load_a(kt - 1 + NST, (kt - 1) % NST);
      load_w(kt - 1 + NST, (kt - 1) % NST);
    }
    cp_async_commit();  // group NST + kt (k-tile kt - 1 + NST when kt >= 1, else empty)
    const uint32_t abase = a_base(kt % NST);
    // SLAB: the k-tile's 64 rows inside the slab (chunk stride NST*64 rows, see w_off)
    const uint32_t bbase = SLAB ? sbase + NST * A_BYTES + (kt % NST) * BK * 128 : abase + A_BYTES;
#pragma unroll
    for (int kk = 0; kk < BK / 16; ++kk) {
      uint32_t af[2][4];
#pragma unroll
      for (int mi = 0; mi < 2; ++mi) {
        const int r = wm * 32 + mi * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int c = kk * 2 + (lane >> 4);
        ldmatrix_x4(abase + r * 128 + swz(r, c) * 16, af[mi][0], af[mi][1], af[mi][2], af[mi][3]);
      }
#pragma unroll
      for (int np = 0; np < NTW / 2; ++np) {
        const int r = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int c = (wn * WN) / 8 + np * 2 + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(bbase + w_off(r, c), b0, b1, b2, b3);
#pragma unroll
        for (int mi = 0; mi < 2; ++mi) {
          mma_bf16_16816(acc[mi][2 * np], af[mi], b0, b1);
          mma_bf16_16816(acc[mi][2 * np + 1], af[mi], b2, b3);
        }
      }
    }
  }
  cp_async_wait<0>();
  if (!w_ok && tid == 0) raise_error(p.err, kErrWaitTimeout);

  // epilogue: scale, bf16 (round to nearest even); rows of empty sequences are zero
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      const int m = m0 + wm * 32 + mi * 16 + (lane >> 2) + h2 * 8;
      if (m >= p.M) continue;
      const int bi = m / p.s, i = m % p.s;
      const float f = (p.seqlens && p.seqlens[bi] == 0) ? 0.f : p.scale;
      __nv_bfloat16* dst = p.c + ((size_t)(bi * p.h + j) * p.s + i) * p.nout + n0 + wn * WN + (lane & 3) * 2;
#pragma unroll
      for (int ni = 0; ni < NTW; ++ni)
        if (n0 + wn * WN + ni * 8 < p.nout)
          *reinterpret_cast<uint32_t*>(dst + ni * 8) = pack_bf16(acc[mi][ni][h2 * 2] * f, acc[mi][ni][h2 * 2 + 1] * f);
    }
}

template <int BM, int BN, int NST, bool TMA_W, bool SLAB = false>
cudaError_t launch_tile(const ProjParams& p, cudaStream_t stream) {
  constexpr int SMEM = NST * (BM * BK * 2 + BK * BN * 2);
  static std::atomic<unsigned long long> smem_limit_set{0};
  if (cudaError_t e = ensure_smem_limit(proj_kernel<BM, BN, NST, TMA_W, SLAB>, SMEM, smem_limit_set)) return e;
  // W viewed as [h * kin rows, nout columns] in 64-column chunks: dims {64 columns, rows,
  // nout/64 chunks}, so one box {64, BK, BN/64} lands chunk-major, [chunk][k row][128 B]
  // swizzled. k-rows of a stage past kin read the next head's rows (their A columns are
  // zero) or zeros past the tensor.
  CUtensorMap tw;
  if (TMA_W) {
    const cuuint64_t dims[3] = {64, (cuuint64_t)p.h * p.kin, (cuuint64_t)p.nout / 64};
    const cuuint64_t strides[2] = {(cuuint64_t)p.nout * 2, 128};
    constexpr int KB = SLAB ? (NST * BK < 256 ? NST * BK : 256) : BK;
    const cuuint32_t box[3] = {64, KB, BN / 64};
    if (!encode_tmap_bf16_sw128(&tw, p.w, 3, dims, strides, box)) return cudaErrorInvalidValue;
  } else {
    memset(&tw, 0, sizeof(tw));
  }
  // programmatic dependent launch: the weight prefetch overlaps the previous kernel
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((p.nout + BN - 1) / BN, (p.M + BM - 1) / BM, p.h);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, proj_kernel<BM, BN, NST, TMA_W, SLAB>, tw, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

// Tile choice: weight-read bound at decode sizes, so the goal is one wave of CTAs with
// every k-stage of a CTA in flight at once, spread evenly over the SMs (absorption with
// d = 128, k = 512, h = 128: 512 CTAs of 32 KB of weight, all resident; 256 CTAs of
// 64 KB left 40 SMs with half the load of the others, 0.6 us slower per call). 32-row tiles when b*s <= 32 (decode with
// one token per sequence), wide column tiles when the weight is wide (absorption:
// d -> k) and narrow ones when it is tall (output projection: k -> d).
cudaError_t launch_proj(const ProjLaunch& a, int num_sms, cudaStream_t stream) {
  ProjParams p;
  p.err = a.err;
  p.wait_ns = a.wait_ns;
  p.a = static_cast<const __nv_bfloat16*>(a.a);
  p.w = static_cast<const __nv_bfloat16*>(a.w);
  p.c = static_cast<__nv_bfloat16*>(a.c);
  p.seqlens = a.seqlens;
  p.b = a.b;
  p.s = a.s;
  p.h = a.h;
  p.kin = a.kin;
  p.nout = a.nout;
  p.M = a.b * a.s;
  p.scale = a.scale;
  (void)num_sms;
  const int kiters = (a.kin + BK - 1) / BK;
  // W by TMA where the output is a whole number of 64-column boxes (the pointer is
  // 16-byte aligned and rows are nout*2 bytes, a multiple of 16, as the API checks)
  const bool tma = a.nout % 64 == 0;
  if (p.M <= 32) {
    if (a.nout >= 256 && kiters <= 2)  // 4 column tiles per head; the weight slab in one box
      return tma ? launch_tile<32, 128, 2, true, true>(p, stream) : launch_tile<32, 128, 2, false>(p, stream);
    if (kiters <= 8)  // every k-stage in flight (96 KB); the weight slab in boxes of 256 rows
      return tma ? launch_tile<32, 64, 8, true, true>(p, stream) : launch_tile<32, 64, 8, false>(p, stream);
    return tma ? launch_tile<32, 64, 4, true>(p, stream) : launch_tile<32, 64, 4, false>(p, stream);
  }
  if (a.nout >= 128)
    return tma ? launch_tile<64, 128, 3, true>(p, stream) : launch_tile<64, 128, 3, false>(p, stream);
  return tma ? launch_tile<64, 64, 3, true>(p, stream) : launch_tile<64, 64, 3, false>(p, stream);
}

}  // namespace decattn
