// Log-sum-exp merge of two attention results over disjoint key sets (sm_103a).
//
// "Mla Analysis" skill page, "MLAvar6+ Design" and "Cost Models - MLAvar6+":
// the hybrid form attends to the o older keys in latent form and to the n
// recent keys in decompressed (expanded) form; the two softmaxes over
// disjoint key sets are joined exactly by their log-sum-exps:
//   lse = log(exp(lse_a) + exp(lse_b)),
//   out = exp(lse_a - lse) out_a + exp(lse_b - lse) out_b.
// A side that saw no key carries lse = -inf and weighs nothing; rows where both
// are -inf get out = 0, lse = -inf. One thread per 8 columns of a row, bf16 in
// (16-byte loads), fp32 weights, bf16 out (round to nearest even). out may be
// the same buffer as out_a or out_b (every element is read before it is written,
// by the same thread).
#include "common.cuh"
#include "internal.h"

namespace decattn {

namespace {

__global__ void __launch_bounds__(256) merge2_kernel(const __nv_bfloat16* __restrict__ oa, const float* __restrict__ la,
                                                     const __nv_bfloat16* __restrict__ ob, const float* __restrict__ lb,
                                                     int rows, int d, __nv_bfloat16* out, float* lse) {
  pdl_wait();  // both results come from earlier kernels on the stream
  pdl_trigger();
  const int per_row = d / 8;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)rows * per_row) return;
  const long long row = idx / per_row;
  const int c = (int)(idx % per_row) * 8;
  const float a = la[row], b = lb[row];
  const float m = fmaxf(a, b);
  float wa = 0.f, wb = 0.f, l = -INFINITY;
  if (m != -INFINITY) {
    const float ea = expf(a - m), eb = expf(b - m);  // exp(-inf) = 0 for an empty side
    const float sum = ea + eb;
    wa = ea / sum;
    wb = eb / sum;
    l = m + logf(sum);
  }
  const uint4 va = *reinterpret_cast<const uint4*>(oa + row * d + c);
  const uint4 vb = *reinterpret_cast<const uint4*>(ob + row * d + c);
  const uint32_t* pa = reinterpret_cast<const uint32_t*>(&va);
  const uint32_t* pb = reinterpret_cast<const uint32_t*>(&vb);
  uint32_t r[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    // an empty side may hold anything (its weight is 0, but 0 * NaN is NaN)
    const float x0 = (wa != 0.f ? wa * bf16_lo(pa[i]) : 0.f) + (wb != 0.f ? wb * bf16_lo(pb[i]) : 0.f);
    const float x1 = (wa != 0.f ? wa * bf16_hi(pa[i]) : 0.f) + (wb != 0.f ? wb * bf16_hi(pb[i]) : 0.f);
    r[i] = pack_bf16(x0, x1);
  }
  *reinterpret_cast<uint4*>(out + row * d + c) = make_uint4(r[0], r[1], r[2], r[3]);
  if (lse && c == 0) lse[row] = l;
}

}  // namespace

cudaError_t launch_merge2(const void* oa, const float* la, const void* ob, const float* lb, int rows, int d, void* out,
                          float* lse, cudaStream_t stream) {
  const long long threads = (long long)rows * (d / 8);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((threads + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, merge2_kernel, static_cast<const __nv_bfloat16*>(oa), la,
                                           static_cast<const __nv_bfloat16*>(ob), lb, rows, d,
                                           static_cast<__nv_bfloat16*>(out), lse);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace decattn
