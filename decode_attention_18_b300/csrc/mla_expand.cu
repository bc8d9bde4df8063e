// Decompressed (expanded-form) MLA cache for sm_103a.
//
// "Mla Analysis" skill page, "Cost Models — FlashAttention" and "Regime
// Selection": the expanded form runs plain per-head attention over keys and
// values rebuilt from the latent cache. For cache row m and head j
//   K[m, j, :] = [ Z[m, :] W_uk[j]^T  ||  K_pe[m, :] ]     (d + p values)
//   V[m, j, :] =   Z[m, :] W_uv[j]                         (d values)
// with the absorbed form's weights (W_uk [h, d, k], W_uv [h, k, d]; the RoPE
// part of the key is shared by all heads). Grouped-head decode with
// Hkv = Hq = h and key / value widths d + p / d then attends over K and V.
//
// The decompression is a dense contraction (M = cache rows, N = h*d, K = k, twice),
// so it runs on the tensor cores. One CTA takes 128 cache rows and a group of heads:
//  * its 128 Z rows (k bf16 each, 128 KB at k = 512) are loaded once by TMA and stay
//    in shared memory as the A operand (K-major, 128-byte swizzle);
//  * the weight blocks of its heads stream through a 4-slot TMA ring: [128 n x 64 k]
//    of W_uk[j] (K-major) and [64 k x 128 n] of W_uv[j] (N-major);
//  * one thread issues tcgen05.mma (M = 128, N = d = 128, K = 16) into one of two TMEM
//    accumulators, so that four epilogue warps drain one output (tcgen05.ld, bf16
//    round to nearest even, 256-byte row stores; the K_pe copy for key outputs) while
//    the next one accumulates.
// Rows past the end read as zeros and are not stored. Every wait is bounded; a wait that
// runs out sets the error word and the CTA winds down (its copies and MMAs waited for).
#include <cstring>

#include "common.cuh"
#include "internal.h"

namespace decattn {

namespace {

constexpr int XM = 128;          // cache rows per CTA (MMA M)
constexpr int XD = 128;          // head dim d (MMA N)
constexpr int XP = 64;           // RoPE dim p copied behind each key
constexpr int XKB = 64;          // k per block (one 128-byte swizzle row)
constexpr int XMAXK = 512;       // largest latent dim
constexpr int XNR = 4;           // weight ring slots
constexpr int XBLK = 16384;      // one [128 x 64] bf16 block
constexpr int XHG = 8;           // heads per CTA
constexpr int XTHREADS = 192;    // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int OFF_A = 0;
constexpr int OFF_RING = OFF_A + (XMAXK / XKB) * XBLK;
constexpr int OFF_BAR = OFF_RING + XNR * XBLK;
enum { X_AFULL = 0, X_FULL = 1, X_EMPTY = X_FULL + XNR, X_ACCF = X_EMPTY + XNR, X_ACCE = X_ACCF + 2, X_FIN = X_ACCE + 2,
       X_NBAR = X_FIN + 1 };
constexpr int XSMEM = OFF_BAR + X_NBAR * 8 + 16 + 1024;  // + tmem slot / abort flag, + alignment slack
constexpr unsigned long long kXTeardownNs = 1000000000ull;

struct ExpandParams {
  const __nv_bfloat16* k_pe;  // [rows, p]
  __nv_bfloat16* k_out;       // [rows, h, d + p]
  __nv_bfloat16* v_out;       // [rows, h, d]
  int rows, h, kl;
  unsigned* err;
  unsigned long long wait_ns;
};

__global__ void __launch_bounds__(XTHREADS, 1)
    mla_expand_kernel(const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_wuk,
                      const __grid_constant__ CUtensorMap tm_wuv, ExpandParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the 128-byte swizzle wants 1024-byte aligned blocks: round the base up (slack reserved)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + X_NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + X_NBAR) + 1;
  const int row0 = blockIdx.x * XM;
  const int j0 = blockIdx.y * XHG;
  const int nh = min(XHG, p.h - j0);
  const int nkb = p.kl / XKB;
  const int nout = 2 * nh;         // outputs: (head, K or V), head-major
  const int nitems = nout * nkb;   // weight blocks through the ring

  if (threadIdx.x == 0) {
    mbar_init(&bars[X_AFULL], 1);
    for (int i = 0; i < XNR; ++i) {
      mbar_init(&bars[X_FULL + i], 1);
      mbar_init(&bars[X_EMPTY + i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[X_ACCF + i], 1);
      mbar_init(&bars[X_ACCE + i], 4);
    }
    mbar_init(&bars[X_FIN], 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_z);
    prefetch_tmap(&tm_wuk);
    prefetch_tmap(&tm_wuv);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 256);
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
  pdl_wait();  // the latent cache may be the previous kernel's output
  pdl_trigger();

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (elect_one()) {
      mbar_expect_tx(&bars[X_AFULL], nkb * XBLK);
      for (int kb = 0; kb < nkb; ++kb) tma_load_2d(sb + OFF_A + kb * XBLK, &tm_z, kb * XKB, row0, &bars[X_AFULL]);
      int last[XNR] = {-1, -1, -1, -1};
      for (int i = 0; i < nitems; ++i) {
        const int slot = i % XNR;
        if (i >= XNR && !mbar_wait(&bars[X_EMPTY + slot], ((i / XNR) - 1) & 1, p.wait_ns, abort_flag)) {
          if (!*abort_flag) fail();
          break;
        }
        const int o = i / nkb, kb = i % nkb;
        const int j = j0 + (o >> 1);
        const uint32_t dst = sb + OFF_RING + slot * XBLK;
        mbar_expect_tx(&bars[X_FULL + slot], XBLK);
        if ((o & 1) == 0)  // W_uk[j] rows n (output columns), k block kb
          tma_load_2d(dst, &tm_wuk, kb * XKB, j * XD, &bars[X_FULL + slot]);
        else  // W_uv[j] rows k (block kb), both 64-column chunks of n
          tma_load_3d(dst, &tm_wuv, 0, j * p.kl + kb * XKB, 0, &bars[X_FULL + slot]);
        last[slot] = i;
      }
      // leave no copy in flight: wait (bounded) for the last one into each slot
      mbar_wait(&bars[X_AFULL], 0, kXTeardownNs, nullptr);
      for (int s = 0; s < XNR; ++s)
        if (last[s] >= 0) mbar_wait(&bars[X_FULL + s], (last[s] / XNR) & 1, kXTeardownNs, nullptr);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (elect_one()) {
      constexpr uint32_t idK = idesc_bf16_f32(XM, XD, false, false);  // B = W_uk[j] rows, K-major
      constexpr uint32_t idV = idesc_bf16_f32(XM, XD, false, true);   // B = W_uv[j] rows, N-major
      const uint64_t da = smem_desc(sb + OFF_A, 16, 1024, kSw128);
      const uint64_t dk = smem_desc(sb + OFF_RING, 16, 1024, kSw128);
      const uint64_t dv = smem_desc(sb + OFF_RING, XKB * 128, 1024, kSw128);  // chunk stride 8 KB
      bool ok = mbar_wait(&bars[X_AFULL], 0, p.wait_ns, abort_flag);
      for (int o = 0; ok && o < nout; ++o) {
        const int buf = o & 1;
        if (o >= 2 && !mbar_wait(&bars[X_ACCE + buf], ((o >> 1) - 1) & 1, p.wait_ns, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_acc = tmem + buf * XD;
        for (int kb = 0; kb < nkb; ++kb) {
          const int i = o * nkb + kb, slot = i % XNR;
          if (!mbar_wait(&bars[X_FULL + slot], (i / XNR) & 1, p.wait_ns, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t a0 = da + (uint64_t)((kb * XBLK) >> 4);
#pragma unroll
          for (int kk = 0; kk < XKB / 16; ++kk) {
            if ((o & 1) == 0)
              tc_mma_ss(d_acc, a0 + 2 * kk, dk + (uint64_t)((slot * XBLK) >> 4) + 2 * kk, idK, (kb | kk) ? 1u : 0u);
            else
              tc_mma_ss(d_acc, a0 + 2 * kk, dv + (uint64_t)((slot * XBLK + kk * 16 * 128) >> 4), idV,
                        (kb | kk) ? 1u : 0u);
          }
          tc_commit(&bars[X_EMPTY + slot]);  // the slot is free once these MMAs have read it
        }
        if (!ok) break;
        tc_commit(&bars[X_ACCF + buf]);
      }
      if (!ok && !*abort_flag) fail();
      // every MMA issued has completed before the accumulators are released
      tc_commit(&bars[X_FIN]);
      mbar_wait(&bars[X_FIN], 0, kXTeardownNs, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ epilogue: TMEM lanes 32*(warp%4) ..
    const int q = warp & 3;
    const int r = q * 32 + lane;  // row within the tile = TMEM lane
    const int row = row0 + r;
    const bool live = row < p.rows;
    for (int o = 0; o < nout; ++o) {
      const int buf = o & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&bars[X_ACCF + buf], (o >> 1) & 1, p.wait_ns, abort_flag))) {
        if (lane == 0 && !*abort_flag) fail();
        break;
      }
      tc_fence_after();
      const int j = j0 + (o >> 1);
      __nv_bfloat16* dst = (o & 1) == 0 ? p.k_out + ((size_t)row * p.h + j) * (XD + XP)
                                        : p.v_out + ((size_t)row * p.h + j) * XD;
#pragma unroll 1
      for (int c = 0; c < XD / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + buf * XD + c * 32, v);
        tmem_ld_wait();
        if (live) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
          for (int u = 0; u < 4; ++u)
            d4[u] = make_uint4(pack_bf16(__uint_as_float(v[8 * u + 0]), __uint_as_float(v[8 * u + 1])),
                               pack_bf16(__uint_as_float(v[8 * u + 2]), __uint_as_float(v[8 * u + 3])),
                               pack_bf16(__uint_as_float(v[8 * u + 4]), __uint_as_float(v[8 * u + 5])),
                               pack_bf16(__uint_as_float(v[8 * u + 6]), __uint_as_float(v[8 * u + 7])));
        }
      }
      if (live && (o & 1) == 0) {  // the shared RoPE part behind the key's d values
        const uint4* src = reinterpret_cast<const uint4*>(p.k_pe + (size_t)row * XP);
        uint4* d4 = reinterpret_cast<uint4*>(dst + XD);
#pragma unroll
        for (int u = 0; u < XP / 8; ++u) d4[u] = __ldg(src + u);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[X_ACCE + buf]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

}  // namespace

bool mla_expand_supported(int d, int k, int p) { return d == XD && p == XP && k >= XKB && k <= XMAXK && k % XKB == 0; }

cudaError_t launch_mla_expand(const ExpandLaunch& a, cudaStream_t stream) {
  static std::atomic<unsigned long long> smem_limit_set{0};
  if (cudaError_t e = ensure_smem_limit(mla_expand_kernel, XSMEM, smem_limit_set)) return e;
  CUtensorMap tz, tuk, tuv;
  {  // Z [rows, k]: boxes [128 rows x 64 k]
    const cuuint64_t dims[2] = {(cuuint64_t)a.k, (cuuint64_t)a.rows};
    const cuuint64_t strides[1] = {(cuuint64_t)a.k * 2};
    const cuuint32_t box[2] = {XKB, XM};
    if (!encode_tmap_bf16_sw128(&tz, a.z, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {  // W_uk as [h*d rows (output columns), k]: boxes [128 rows x 64 k]
    const cuuint64_t dims[2] = {(cuuint64_t)a.k, (cuuint64_t)a.h * XD};
    const cuuint64_t strides[1] = {(cuuint64_t)a.k * 2};
    const cuuint32_t box[2] = {XKB, XD};
    if (!encode_tmap_bf16_sw128(&tuk, a.w_uk, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {  // W_uv as [h*k rows, d] in 64-column chunks: boxes {64, 64 rows, 2 chunks}, chunk-major
    const cuuint64_t dims[3] = {64, (cuuint64_t)a.h * a.k, XD / 64};
    const cuuint64_t strides[2] = {(cuuint64_t)XD * 2, 128};
    const cuuint32_t box[3] = {64, XKB, XD / 64};
    if (!encode_tmap_bf16_sw128(&tuv, a.w_uv, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  ExpandParams p;
  p.k_pe = static_cast<const __nv_bfloat16*>(a.k_pe);
  p.k_out = static_cast<__nv_bfloat16*>(a.k_out);
  p.v_out = static_cast<__nv_bfloat16*>(a.v_out);
  p.rows = a.rows;
  p.h = a.h;
  p.kl = a.k;
  p.err = a.err;
  p.wait_ns = a.wait_ns;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.rows + XM - 1) / XM, (a.h + XHG - 1) / XHG, 1);
  cfg.blockDim = dim3(XTHREADS);
  cfg.dynamicSmemBytes = XSMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, mla_expand_kernel, tz, tuk, tuv, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace decattn
