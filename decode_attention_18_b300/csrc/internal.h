// Internal launch interfaces between the C-ABI layer (api.cu) and the kernel
// translation units. Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace decattn {

struct GqaLaunch {
  const void* q;
  const void* k;
  const void* v;
  const int32_t* seqlens;
  const int32_t* block_table;
  int max_pages, paged, capacity, num_pages;
  int b, s, hq, hkv;
  int dk, dv;  // query/key width, value/output width
  int fp8;     // cache in e4m3 bytes, dequantised as k_scale * K and v_scale * V
  float k_scale, v_scale;
  int nsplit, chunk;
  float scale;
  void* out;
  float* lse;
  float* ws_o;    // [b*hq*s, nsplit, dv] (nsplit > 1), or balanced: [records, rows per CTA, dv]
  float* ws_lse;  // [b*hq*s, nsplit], or balanced: [records, rows per CTA]
  int* meta;      // balanced: [work items][2] {first record, count}
  int balanced_grid;  // > 0: balanced schedule over this many CTAs
  unsigned* err;
  unsigned long long wait_ns;  // limit of the bounded tile waits
  int test_timeout;            // forced-timeout test: one wait on a barrier nothing signals
};

// rows of one grouped-head CTA (multiple of 16) for `rows` query rows per KV head
int gqa_rows_per_cta(int rows);
int gqa_ctas_per_sm(int dk, int dv);
int gqa_balanced_ctas_per_sm(int dk, int dv, int rows, bool fp8);  // measured occupancy of the balanced kernel
bool gqa_supported(int dk, int dv, bool fp8);
cudaError_t launch_gqa(const GqaLaunch& p, cudaStream_t stream);
// tensor-core grouped-head kernel for KV heads with many query rows (no split: one CTA
// per 128 query rows of a KV head, every key in one pass)
bool gqa_prefill_supported(int dk, int dv, bool fp8);
cudaError_t launch_gqa_prefill(const GqaLaunch& p, cudaStream_t stream);

// log-sum-exp merge of split partials: rows x nsplit partials of width d (fp32, or bf16
// when bf16_partials) and their fp32 LSEs
cudaError_t launch_combine(const void* ws_o, bool bf16_partials, const float* ws_lse, const int32_t* seqlens, int rows,
                           int rows_per_seq, int nsplit, int chunk, int d, void* out, float* lse, cudaStream_t stream);
// combine of the latent kernel's tail split: tail_units * 128 partial rows of k bf16
// partials each (unit tail_whole + i, rows i * 128 ..), merged into their rows of out
cudaError_t launch_combine_tail(const void* ws_o, const float* ws_lse, const int32_t* seqlens, int tail_units,
                                int tail_whole, int mtiles, int rows_per_seq, int k, int chunk, int d, void* out,
                                float* lse, cudaStream_t stream);
// combine of the balanced grouped-head schedules (gqa_balanced_kernel, rpb = its rows per
// CTA; the tensor-core kernel's balanced split, rpb = 128): records [records][rpb][d]
cudaError_t launch_combine_balanced(const float* ws_o, const float* ws_lse, const int* meta, const int32_t* seqlens,
                                    int b, int hq, int s, int hkv, int d, int rpb, long long records, void* out,
                                    float* lse, cudaStream_t stream);

struct ProjLaunch {
  unsigned* err;     // device error word
  unsigned long long wait_ns;
  const void* a;     // [b, h, s, kin]
  const void* w;     // [h, kin, nout]
  void* c;           // [b, h, s, nout]
  const int32_t* seqlens;
  int b, s, h, kin, nout;
  float scale;
};
cudaError_t launch_proj(const ProjLaunch& p, int num_sms, cudaStream_t stream);

struct MlaLaunch {
  const void* qz;
  const void* q_pe;
  const void* z;
  const void* k_pe;
  const int32_t* seqlens;
  const int32_t* block_table;
  int max_pages, paged, capacity, num_pages;
  int b, s, h, k, p;
  int nsplit, chunk;
  float scale;
  void* o_lat;
  float* lse;
  void* ws_o;     // [b*h*s, nsplit, k] bf16 O / l partials (tail split: [tail rows, tail_k, k])
  float* ws_lse;  // [b*h*s, nsplit] (tail split: [tail rows, tail_k])
  int tail_whole, tail_units, tail_k, tail_chunk;  // tail split (tail_k > 0): whole units, split units
  unsigned* err;
  unsigned long long wait_ns;
  int test_timeout;
};
// out = LSE-weighted merge of two results over disjoint key sets (rows x d, bf16; fp32 LSEs)
cudaError_t launch_merge2(const void* oa, const float* la, const void* ob, const float* lb, int rows, int d, void* out,
                          float* lse, cudaStream_t stream);

// Expanded-form MLA cache: K = [Z W_uk^T || K_pe], V = Z W_uv for `rows` cache rows
struct ExpandLaunch {
  const void* z;     // [rows, k]
  const void* k_pe;  // [rows, p]
  const void* w_uk;  // [h, d, k]
  const void* w_uv;  // [h, k, d]
  void* k_out;       // [rows, h, d + p]
  void* v_out;       // [rows, h, d]
  int rows, h, k;
  unsigned* err;
  unsigned long long wait_ns;
};
bool mla_expand_supported(int d, int k, int p);
cudaError_t launch_mla_expand(const ExpandLaunch& p, cudaStream_t stream);

// CTAs per 128-row tile of the latent kernel (a cluster: scores CTA + output CTA)
int mla_ctas_per_row_tile();
// keys per latent tile (context chunks are multiples of it)
int mla_tile_keys();
bool mla_supported(int k, int p);
cudaError_t launch_mla_latent(const MlaLaunch& p, cudaStream_t stream);

}  // namespace decattn
