// Per-head projection GEMMs of the absorbed MLA pipeline (sm_103a).
//
// "Mla Analysis" skill page, "Absorption Trick (FlashMLA)": the score line
// folds the key up-projection into the query (Qz = q_nope W_uk, one GEMM per
// head) and the value line leaves the latent output to be decompressed by a
// separate kernel (O = O_lat W_uv). Both are batched per-head GEMMs
//   C[b, j, r, :] = scale * A[b, j, r, :] @ W[j]      (W[j] is kin x nout)
// with M = b*s rows per head. At decode sizes M is small (32 rows for 32
// sequences of one token) and the kernel is bound by reading W (h*kin*nout
// bf16, 16.8 MB for h=128, d=128, k=512), so it streams W once through a
// cp.async pipeline and runs mma.sync m16n8k16 (bf16, fp32 accumulate).
#include "common.cuh"
#include "internal.h"

namespace decattn {

namespace {

constexpr int BK = 64;

struct ProjParams {
  const __nv_bfloat16* a;
  const __nv_bfloat16* w;
  __nv_bfloat16* c;
  const int32_t* seqlens;
  int b, s, h, kin, nout, M;
  float scale;
};

__device__ __forceinline__ uint32_t swz(int row, int chunk) { return (uint32_t)(chunk ^ (row & 7)); }

// One CTA: BM rows of one head x BN output columns, 4 warps laid out (BM/32) x (4/(BM/32)),
// each warp 32 rows x WN columns; NST k-stages of BK in flight (cp.async, 16-byte chunks).
template <int BM, int BN, int NST>
__global__ void __launch_bounds__(128) proj_kernel(ProjParams p) {
  constexpr int WMW = BM / 32;               // warps along M
  constexpr int WNW = 4 / WMW;               // warps along N
  constexpr int WN = BN / WNW;               // columns per warp
  constexpr int NTW = WN / 8;                // n-tiles per warp
  constexpr int A_BYTES = BM * BK * 2;       // [BM rows][64 k], rows of 128 B
  constexpr int B_ROW = BN * 2;              // bytes per k row of the W tile
  constexpr int B_BYTES = BK * B_ROW;        // [64 k][BN n]
  constexpr int STAGE = A_BYTES + B_BYTES;
  static_assert(NTW % 2 == 0 && (BM * 8) % 128 == 0 && (BK * (BN / 8)) % 128 == 0, "tile shape");
  extern __shared__ __align__(1024) uint8_t smem[];

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

  auto load_a = [&](int kt, int stage) {
    const uint32_t adst = sbase + stage * STAGE;
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
  auto load_w = [&](int kt, int stage) {
    const uint32_t bdst = sbase + stage * STAGE + A_BYTES;
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

  // The weight does not come from the previous kernel in the stream: its first stages
  // are requested before pdl_wait, so they load while that kernel finishes. (They join
  // the first commit group, whose completion is awaited before stage 0 is used.)
#pragma unroll
  for (int t = 0; t < NST - 1; ++t)
    if (t < kiters) load_w(t, t);
  pdl_wait();  // the activations (and lengths) are the previous kernel's results
  pdl_trigger();
#pragma unroll
  for (int t = 0; t < NST - 1; ++t) {
    if (t < kiters) load_a(t, t);
    cp_async_commit();
  }
  for (int kt = 0; kt < kiters; ++kt) {
    cp_async_wait<NST - 2>();
    __syncthreads();
    if (kt + NST - 1 < kiters) {
      load_a(kt + NST - 1, (kt + NST - 1) % NST);
      load_w(kt + NST - 1, (kt + NST - 1) % NST);
    }
    cp_async_commit();
    const uint32_t abase = sbase + (kt % NST) * STAGE;
    const uint32_t bbase = abase + A_BYTES;
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
        ldmatrix_x4_trans(bbase + r * B_ROW + swz(r, c) * 16, b0, b1, b2, b3);
#pragma unroll
        for (int mi = 0; mi < 2; ++mi) {
          mma_bf16_16816(acc[mi][2 * np], af[mi], b0, b1);
          mma_bf16_16816(acc[mi][2 * np + 1], af[mi], b2, b3);
        }
      }
    }
  }
  cp_async_wait<0>();

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

template <int BM, int BN, int NST>
cudaError_t launch_tile(const ProjParams& p, cudaStream_t stream) {
  constexpr int SMEM = NST * (BM * BK * 2 + BK * BN * 2);
  static std::atomic<unsigned long long> smem_limit_set{0};
  if (cudaError_t e = ensure_smem_limit(proj_kernel<BM, BN, NST>, SMEM, smem_limit_set)) return e;
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
  const cudaError_t e = cudaLaunchKernelEx(&cfg, proj_kernel<BM, BN, NST>, p);
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
  if (p.M <= 32) {
    if (a.nout >= 256 && kiters <= 2) return launch_tile<32, 128, 2>(p, stream);  // 4 column tiles per head
    if (kiters <= 8) return launch_tile<32, 64, 8>(p, stream);  // every k-stage in flight (96 KB)
    return launch_tile<32, 64, 4>(p, stream);
  }
  if (a.nout >= 128) return launch_tile<64, 128, 3>(p, stream);
  return launch_tile<64, 64, 3>(p, stream);
}

}  // namespace decattn
