// C ABI of the decode-attention library: argument checks, the split planner,
// workspace sizing, the device error word and the launches. Every entry point
// returns a status and enqueues on the caller's stream; nothing here
// allocates device memory or synchronises (except decattn_check_errors).
#include <atomic>
#include <climits>
#include <cstdint>
#include <mutex>

#include "decattn.h"
#include "common.cuh"
#include "internal.h"

namespace decattn {
namespace {

// device error word (bit flags set by the kernels, read by decattn_check_errors)
__device__ unsigned g_err_word;

struct DeviceState {
  bool ready = false;
  unsigned* err = nullptr;
  int sms = 0;
};
constexpr int kMaxDevices = 64;
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;

std::atomic<unsigned long long> g_wait_ns{0};
std::atomic<int> g_forced_splits{0};
std::atomic<int> g_last_splits{0};
std::atomic<int> g_test_timeout{0};
std::atomic<int> g_grouped_kernel{0};  // 0 auto, 1 split-KV kernels, 2 tensor-core kernel (where the widths allow)

constexpr unsigned long long kDefaultWaitNs = 2000000000ull;  // 2 s
constexpr int kPage = 64;  // chunks are whole 64-key pages (and whole kernel tiles)

// Per-device set-up on first use: the error word's device address and the SM count.
int device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DECATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_err_word) != cudaSuccess) return DECATTN_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
      return DECATTN_ERR_CUDA;
    st.err = static_cast<unsigned*>(addr);
    st.sms = sms;
    st.ready = true;
  }
  *out = &st;
  return DECATTN_OK;
}

unsigned long long wait_limit() {
  const unsigned long long w = g_wait_ns.load();
  return w ? w : kDefaultWaitNs;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

constexpr int kMaxS = 1024;  // new tokens per sequence in one call (decode, speculative and prefill-sized)

struct Plan {
  int nsplit;
  int chunk;
};

// Split planner: pick the number of context chunks. base = CTAs per chunk index
// (sequences x heads x row blocks), slots = CTAs resident on the whole GPU at once,
// align = chunk granularity (a multiple of the 64-key page and of the kernel's key
// tile). Cost model, in keys of one CTA's work:
//   waves x (chunk + overhead) + (nsplit > 1 ? combine : 0)
// overhead = a CTA's prologue (pipeline fill, query load, epilogue), combine = the
// second kernel and the partials' round trip. Measured on B300 (b=32, 8 KV heads,
// d=128, 4096 keys): unsplit runs at 95% of HBM bandwidth, 8 chunks at 67%.
Plan plan_splits(long long base, int max_seqlen, long long slots, int overhead_keys, int combine_keys, int align) {
  Plan pl{1, align};
  const long long L = max_seqlen > 0 ? max_seqlen : 1;
  const int max_n = (int)ceil_div(L, align);
  auto chunk_for = [&](int n) { return (int)(ceil_div(ceil_div(L, n), align) * align); };
  const int forced = g_forced_splits.load();
  if (forced > 0) {
    const int n = forced < max_n ? forced : max_n;
    pl.chunk = chunk_for(n);
    pl.nsplit = (int)ceil_div(L, pl.chunk);
    return pl;
  }
  double best = 1e300;
  for (int n = 1; n <= max_n && n <= 1024; ++n) {
    const int chunk = chunk_for(n);
    const int ne = (int)ceil_div(L, chunk);
    if (ne != n) continue;
    const long long waves = ceil_div(base * ne, slots);
    const double cost = (double)waves * (chunk + overhead_keys) + (ne > 1 ? combine_keys : 0);
    if (cost < best * 0.999) {
      best = cost;
      pl.nsplit = ne;
      pl.chunk = chunk;
    }
  }
  return pl;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// split partials: O [rows, nsplit, width] of elem_bytes each, then LSE [rows, nsplit] fp32
size_t partial_bytes(long long rows, int nsplit, int width, size_t elem_bytes = sizeof(float)) {
  if (nsplit <= 1) return 0;
  return align256((size_t)rows * nsplit * width * elem_bytes) + align256((size_t)rows * nsplit * sizeof(float));
}
constexpr size_t kMlaPartialBytes = 2;  // the latent kernel's O / l partials are bf16

int check_kv(const decattn_kv& kv, int b, int max_seqlen) {
  if (kv.paged) {
    if (!kv.block_table || kv.page_size != 64 || kv.num_pages < 1 || kv.max_pages < 1) return DECATTN_ERR_INVALID_ARG;
    if ((long long)kv.max_pages * 64 < max_seqlen) return DECATTN_ERR_INVALID_ARG;
    if ((long long)kv.num_pages * 64 > INT_MAX) return DECATTN_ERR_INVALID_ARG;
  } else {
    if (kv.capacity < max_seqlen || kv.capacity < 1) return DECATTN_ERR_INVALID_ARG;
    if ((long long)b * kv.capacity > INT_MAX) return DECATTN_ERR_INVALID_ARG;
  }
  return DECATTN_OK;
}

// --- grouped-head plan
Plan gqa_plan(int b, int s, int hq, int hkv, int dk, int dv, int max_seqlen, int sms) {
  const int rows = (hq / hkv) * s;
  const long long base = (long long)b * hkv * ceil_div(rows, gqa_rows_per_cta(rows));
  const long long slots = (long long)sms * gqa_ctas_per_sm(dk, dv);
  return plan_splits(base, max_seqlen, slots, 256, 512, kPage);
}

// Balanced grouped-head schedule (gqa_balanced_kernel): used when the planner splits
// the context, no split count is forced and a CTA holds one 16-row m-tile (the
// tensor-core variant keeps the fixed chunks). Its grid is one wave of CTAs; the
// per-CTA share of the key tiles is computed on the device from the actual lengths.
// With two m-tiles (more than 16 query rows per KV head) the register-bound main loop
// measured ~12 % slower per tile inside the balanced kernel on B300 (24-head MQA,
// d = 256: 2.01 vs 1.79 us per 64-key tile, clocks at maximum in both), more than the
// balance wins back, so those shapes keep the fixed chunks.
struct GqaBalanced {
  int grid = 0;          // 0: fixed chunks
  long long items = 0;   // work items (sequence, KV head, row block)
  int rpb = 0;           // rows per CTA
};
GqaBalanced gqa_balanced(const Plan& pl, int b, int s, int hq, int hkv, int dk, int dv, int sms, bool fp8 = false) {
  GqaBalanced gb;
  const int rows = (hq / hkv) * s;
  if (pl.nsplit <= 1 || g_forced_splits.load() > 0 || gqa_rows_per_cta(rows) > 16) return gb;
  gb.rpb = gqa_rows_per_cta(rows);
  gb.items = (long long)b * hkv * ceil_div(rows, gb.rpb);
  gb.grid = sms * gqa_balanced_ctas_per_sm(dk, dv, rows, fp8);
  return gb;
}
size_t balanced_bytes(const GqaBalanced& gb, int dv) {
  const long long records = gb.items + gb.grid;
  return align256((size_t)records * gb.rpb * dv * sizeof(float)) + align256((size_t)records * gb.rpb * sizeof(float)) +
         align256((size_t)gb.items * 2 * sizeof(int));
}

// --- latent MLA plan: one cluster of two CTAs (each alone on its SM) per (sequence,
// 128-row tile, chunk), so sms / 2 clusters run at once
Plan mla_plan(int b, int s, int h, int k, int max_seqlen, int sms) {
  (void)k;
  const long long base = (long long)b * ceil_div((long long)h * s, 128);
  const int per = mla_ctas_per_row_tile();
  return plan_splits(base, max_seqlen, sms / per > 0 ? sms / per : 1, 384, 512, mla_tile_keys());
}
// Tail split: with one chunk per (sequence, row tile) unit and U units on P cluster slots,
// the last wave holds only U mod P units. Those units are cut into k = P / (U mod P) >= 2
// chunks each, so that the last wave runs k times shorter; the other units stay whole.
struct MlaTail {
  int whole = 0, units = 0, k = 0, chunk = 0;
};
MlaTail mla_tail(int b, int s, int h, int max_seqlen, int sms, const Plan& pl) {
  MlaTail t;
  if (g_forced_splits.load() > 0 || pl.nsplit != 1 || max_seqlen <= 0) return t;
  const long long U = (long long)b * ceil_div((long long)h * s, 128);
  const long long P = sms / mla_ctas_per_row_tile();
  if (P <= 0 || U <= P) return t;
  const long long rm = U % P;
  if (rm == 0 || P / rm < 2 || U > INT_MAX) return t;
  const int k = (int)(P / rm);
  const int tk = mla_tile_keys();
  const int chunk = (int)(ceil_div(ceil_div(max_seqlen, k), tk) * tk);
  if (chunk >= max_seqlen) return t;
  t.whole = (int)(U - rm);
  t.units = (int)rm;
  t.k = k;
  t.chunk = chunk;
  return t;
}
size_t mla_tail_bytes(const MlaTail& t, int k_lat) {
  if (t.k == 0) return 0;
  const size_t rows = (size_t)t.units * 128 * t.k;
  return align256(rows * k_lat * kMlaPartialBytes) + align256(rows * sizeof(float));
}

}  // namespace
}  // namespace decattn

namespace decattn {
namespace {

// KV heads with many query rows (prefill-sized s, large groups) run the tensor-core kernel:
// one pass over the keys per 128 rows, no split, no workspace (a forced split count keeps
// the split-KV kernels, which is what it is for)
// Auto: the tensor-core kernel from 32 query rows per KV head with values 128 wide (below
// 32 rows the split-KV kernel's 16-row tiles keep up with HBM: 0.94 vs 0.87 of it at 16
// rows of the expanded form; at 256-wide rows only two 64 KB stages fit beside Q and P,
// and the 24-row MQA shape measured 80 vs 61 us, so those keep the split-KV kernels).
// Automatic choice, from same-box graph-replay measurements of both kernels (rows R =
// query rows per KV head): 192 / 128 (expanded MLA) from R = 1 up (s = 1: 1723 vs 1742 us,
// s = 16: 1747 vs 1925, s = 128: 1747 vs 8632); 256 / 256 from R = 24 (ragged paged MQA:
// 54 vs 60 us; R = 48: 51 vs 76; over an FP8 cache 45 vs 64 us, and at R = 6 144 vs 127);
// 128 / 128 from R = 32 (R = 16: 123 vs 86 us; R = 32: 121 vs 133). Below those the
// split-KV mma.sync kernel's 16-row tiles waste less.
bool use_prefill(int b, int hq, int hkv, int s, int dk, int dv, bool fp8, int sms) {
  (void)b;
  (void)sms;
  if (!gqa_prefill_supported(dk, dv, fp8)) return false;
  const int mode = g_grouped_kernel.load();
  if (mode == 1) return false;
  if (mode == 2) return true;
  const long long rows = (long long)(hq / hkv) * s;
  if (dk == 192) return true;
  return rows >= (dk == 256 ? 24 : 32);
}

// the tensor-core kernel's context split: one CTA per SM, 128 rows per CTA
Plan prefill_plan(int b, int s, int hq, int hkv, int max_seqlen, int sms) {
  const long long rows = (long long)(hq / hkv) * s;
  const long long base = (long long)b * hkv * ceil_div(rows, 128);
  return plan_splits(base, max_seqlen, sms, 256, 512, kPage);
}
// Its balanced split (planned on the device from the actual lengths) whenever the work
// items are fewer than the CTAs of one wave and no split count is forced; 0: fixed chunks.
long long prefill_items(int b, int s, int hq, int hkv) {
  return (long long)b * hkv * ceil_div((long long)(hq / hkv) * s, 128);
}
int prefill_balanced_grid(int b, int s, int hq, int hkv, int sms) {
  if (g_forced_splits.load() > 0) return 0;
  return prefill_items(b, s, hq, hkv) < sms ? sms : 0;
}
size_t prefill_balanced_bytes(int b, int s, int hq, int hkv, int dv, int grid) {
  return align256((size_t)grid * 128 * dv * sizeof(float)) + align256((size_t)grid * 128 * sizeof(float)) +
         align256((size_t)prefill_items(b, s, hq, hkv) * 2 * sizeof(int));
}

size_t gqa_workspace(int b, int s, int hq, int hkv, int dk, int dv, int max_seqlen, bool fp8) {
  if (b < 1 || s < 1 || hq < 1 || hkv < 1 || hq % hkv || dk < 1 || dv < 1) return 0;
  DeviceState* st = nullptr;
  if (device_state(&st)) return 0;
  if (use_prefill(b, hq, hkv, s, dk, dv, fp8, st->sms)) {
    if (const int grid = prefill_balanced_grid(b, s, hq, hkv, st->sms)) return prefill_balanced_bytes(b, s, hq, hkv, dv, grid);
    return partial_bytes((long long)b * hq * s, prefill_plan(b, s, hq, hkv, max_seqlen, st->sms).nsplit, dv);
  }
  const Plan pl = gqa_plan(b, s, hq, hkv, dk, dv, max_seqlen, st->sms);
  const GqaBalanced gb = gqa_balanced(pl, b, s, hq, hkv, dk, dv, st->sms, fp8);
  if (gb.grid > 0) return balanced_bytes(gb, dv);
  return partial_bytes((long long)b * hq * s, pl.nsplit, dv);
}

// grouped-head decode, bf16 or FP8 (e4m3 bytes with per-tensor scales) cache
int gqa_decode_impl(const void* q, const void* k, const void* v, decattn_kv kv, const int32_t* seqlens, int max_seqlen,
                    int b, int s, int hq, int hkv, int dk, int dv, float scale, bool fp8, float k_scale,
                    float v_scale, void* out, float* lse, void* workspace, size_t workspace_bytes,
                    cudaStream_t stream) {
  if (b < 0 || s < 1 || s > kMaxS || hq < 1 || hkv < 1 || hq % hkv || max_seqlen < 0) return DECATTN_ERR_INVALID_ARG;
  if (b == 0) return DECATTN_OK;
  if (!q || !k || !v || !seqlens || !out) return DECATTN_ERR_INVALID_ARG;
  if (fp8 && !(k_scale > 0.f && v_scale > 0.f && k_scale < INFINITY && v_scale < INFINITY))
    return DECATTN_ERR_INVALID_ARG;
  if (!gqa_supported(dk, dv, fp8)) return DECATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return DECATTN_ERR_INVALID_ARG;
  if (hkv > 65535 || b > 65535) return DECATTN_ERR_INVALID_ARG;
  if (int rc = check_kv(kv, b, max_seqlen)) return rc;
  DeviceState* st = nullptr;
  if (int rc = device_state(&st)) return rc;
  if (use_prefill(b, hq, hkv, s, dk, dv, fp8, st->sms)) {
    if ((long long)b * hq * s > INT_MAX / 2) return DECATTN_ERR_INVALID_ARG;
    const Plan pp = prefill_plan(b, s, hq, hkv, max_seqlen, st->sms);
    const long long prow = (long long)b * hq * s;
    const int bgrid = prefill_balanced_grid(b, s, hq, hkv, st->sms);
    const size_t pneed = bgrid > 0 ? prefill_balanced_bytes(b, s, hq, hkv, dv, bgrid) : partial_bytes(prow, pp.nsplit, dv);
    if (pneed > 0 && (!workspace || workspace_bytes < pneed || !aligned16(workspace))) return DECATTN_ERR_WORKSPACE;
    if ((long long)pp.nsplit * ceil_div((long long)(hq / hkv) * s, 128) > INT_MAX) return DECATTN_ERR_INVALID_ARG;
    GqaLaunch a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.seqlens = seqlens;
    a.block_table = kv.block_table;
    a.max_pages = kv.max_pages;
    a.paged = kv.paged;
    a.capacity = kv.capacity;
    a.num_pages = kv.num_pages;
    a.b = b;
    a.s = s;
    a.hq = hq;
    a.hkv = hkv;
    a.dk = dk;
    a.dv = dv;
    a.fp8 = fp8 ? 1 : 0;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.nsplit = pp.nsplit;
    a.chunk = pp.chunk;
    a.scale = scale;
    a.out = out;
    a.lse = lse;
    a.ws_o = pp.nsplit > 1 ? static_cast<float*>(workspace) : nullptr;
    a.ws_lse = pp.nsplit > 1 ? reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                                         align256((size_t)prow * pp.nsplit * dv * sizeof(float)))
                             : nullptr;
    a.meta = nullptr;
    a.balanced_grid = bgrid;
    if (bgrid > 0) {
      char* w = static_cast<char*>(workspace);
      const size_t o_bytes = align256((size_t)bgrid * 128 * dv * sizeof(float));
      a.ws_o = reinterpret_cast<float*>(w);
      a.ws_lse = reinterpret_cast<float*>(w + o_bytes);
      a.meta = reinterpret_cast<int*>(w + o_bytes + align256((size_t)bgrid * 128 * sizeof(float)));
    }
    a.err = st->err;
    a.wait_ns = wait_limit();
    a.test_timeout = g_test_timeout.load();
    g_last_splits.store(bgrid > 0 ? 0 : pp.nsplit);  // 0: pieces planned on the device
    if (launch_gqa_prefill(a, stream) != cudaSuccess) return DECATTN_ERR_CUDA;
    if (bgrid > 0) {
      if (launch_combine_balanced(a.ws_o, a.ws_lse, a.meta, seqlens, b, hq, s, hkv, dv, 128, bgrid, out, lse,
                                  stream) != cudaSuccess)
        return DECATTN_ERR_CUDA;
    } else if (pp.nsplit > 1 && launch_combine(a.ws_o, false, a.ws_lse, seqlens, (int)prow, hq * s, pp.nsplit,
                                               pp.chunk, dv, out, lse, stream) != cudaSuccess) {
      return DECATTN_ERR_CUDA;
    }
    return DECATTN_OK;
  }
  const Plan pl = gqa_plan(b, s, hq, hkv, dk, dv, max_seqlen, st->sms);
  const GqaBalanced gb = gqa_balanced(pl, b, s, hq, hkv, dk, dv, st->sms, fp8);
  const long long rows = (long long)b * hq * s;
  const size_t need = gb.grid > 0 ? balanced_bytes(gb, dv) : partial_bytes(rows, pl.nsplit, dv);
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace))) return DECATTN_ERR_WORKSPACE;
  GqaLaunch a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.seqlens = seqlens;
  a.block_table = kv.block_table;
  a.max_pages = kv.max_pages;
  a.paged = kv.paged;
  a.capacity = kv.capacity;
  a.num_pages = kv.num_pages;
  a.b = b;
  a.s = s;
  a.hq = hq;
  a.hkv = hkv;
  a.dk = dk;
  a.dv = dv;
  a.fp8 = fp8 ? 1 : 0;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.nsplit = pl.nsplit;
  a.chunk = pl.chunk;
  a.scale = scale;
  a.out = out;
  a.lse = lse;
  a.ws_o = pl.nsplit > 1 ? static_cast<float*>(workspace) : nullptr;
  a.ws_lse = pl.nsplit > 1 ? reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                                       align256((size_t)rows * pl.nsplit * dv * sizeof(float)))
                           : nullptr;
  a.meta = nullptr;
  a.balanced_grid = gb.grid;
  if (gb.grid > 0) {
    const long long records = gb.items + gb.grid;
    char* w = static_cast<char*>(workspace);
    const size_t o_bytes = align256((size_t)records * gb.rpb * dv * sizeof(float));
    a.ws_o = reinterpret_cast<float*>(w);
    a.ws_lse = reinterpret_cast<float*>(w + o_bytes);
    a.meta = reinterpret_cast<int*>(w + o_bytes + align256((size_t)records * gb.rpb * sizeof(float)));
  }
  a.err = st->err;
  a.wait_ns = wait_limit();
  a.test_timeout = g_test_timeout.load();
  g_last_splits.store(pl.nsplit);
  if (launch_gqa(a, stream) != cudaSuccess) return DECATTN_ERR_CUDA;
  if (gb.grid > 0) {
    if (launch_combine_balanced(a.ws_o, a.ws_lse, a.meta, seqlens, b, hq, s, hkv, dv, gb.rpb, gb.items + gb.grid,
                                out, lse, stream) != cudaSuccess)
      return DECATTN_ERR_CUDA;
  } else if (pl.nsplit > 1) {
    if (launch_combine(a.ws_o, false, a.ws_lse, seqlens, (int)rows, hq * s, pl.nsplit, pl.chunk, dv, out, lse,
                       stream) != cudaSuccess)
      return DECATTN_ERR_CUDA;
  }
  return DECATTN_OK;
}

}  // namespace
}  // namespace decattn

using namespace decattn;

extern "C" {

const char* decattn_status_string(int status) {
  switch (status) {
    case DECATTN_OK: return "ok";
    case DECATTN_ERR_INVALID_ARG: return "invalid argument";
    case DECATTN_ERR_UNSUPPORTED: return "unsupported shape (no compiled instance)";
    case DECATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case DECATTN_ERR_CUDA: return "CUDA runtime error";
    case DECATTN_ERR_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

void decattn_set_wait_limit_ns(unsigned long long ns) { g_wait_ns.store(ns); }
void decattn_set_forced_splits(int nsplit) { g_forced_splits.store(nsplit > 0 ? nsplit : 0); }
int decattn_last_num_splits(void) { return g_last_splits.load(); }
void decattn_test_force_timeout(int on) { g_test_timeout.store(on ? 1 : 0); }
void decattn_set_grouped_kernel(int mode) { g_grouped_kernel.store(mode == 1 || mode == 2 ? mode : 0); }

int decattn_check_errors(cudaStream_t stream) {
  DeviceState* st = nullptr;
  int rc = device_state(&st);
  if (rc) return rc;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return DECATTN_ERR_CUDA;
  unsigned word = 0;
  if (cudaMemcpyFromSymbol(&word, g_err_word, sizeof(word)) != cudaSuccess) return DECATTN_ERR_CUDA;
  const unsigned zero = 0;
  if (cudaMemcpyToSymbol(g_err_word, &zero, sizeof(zero)) != cudaSuccess) return DECATTN_ERR_CUDA;
  if (word & kErrWaitTimeout) return DECATTN_ERR_TIMEOUT;
  if (word & kErrBadPage) return DECATTN_ERR_INVALID_ARG;
  if (word & kErrLaunch) return DECATTN_ERR_CUDA;
  return DECATTN_OK;
}

// ------------------------------------------------------------------ grouped-head


size_t gqa_decode_workspace_size(int b, int s, int hq, int hkv, int d, int max_seqlen) {
  return gqa_workspace(b, s, hq, hkv, d, d, max_seqlen, false);
}

size_t gqa_decode_dv_workspace_size(int b, int s, int hq, int hkv, int dk, int dv, int max_seqlen) {
  return gqa_workspace(b, s, hq, hkv, dk, dv, max_seqlen, false);
}

size_t gqa_decode_fp8_workspace_size(int b, int s, int hq, int hkv, int d, int max_seqlen) {
  return gqa_workspace(b, s, hq, hkv, d, d, max_seqlen, true);
}

int gqa_decode_dv(const decattn_bf16* q, const decattn_bf16* k, const decattn_bf16* v, decattn_kv kv,
                  const int32_t* seqlens, int max_seqlen, int b, int s, int hq, int hkv, int dk, int dv, float scale,
                  decattn_bf16* out, float* lse, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return gqa_decode_impl(q, k, v, kv, seqlens, max_seqlen, b, s, hq, hkv, dk, dv, scale, false, 1.f, 1.f, out, lse,
                         workspace, workspace_bytes, stream);
}

int gqa_decode_fp8(const decattn_bf16* q, const uint8_t* k, const uint8_t* v, decattn_kv kv, const int32_t* seqlens,
                   int max_seqlen, int b, int s, int hq, int hkv, int d, float scale, float k_scale, float v_scale,
                   decattn_bf16* out, float* lse, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return gqa_decode_impl(q, k, v, kv, seqlens, max_seqlen, b, s, hq, hkv, d, d, scale, true, k_scale, v_scale, out,
                         lse, workspace, workspace_bytes, stream);
}

int gqa_decode(const decattn_bf16* q, const decattn_bf16* k, const decattn_bf16* v, decattn_kv kv,
               const int32_t* seqlens, int max_seqlen, int b, int s, int hq, int hkv, int d, float scale,
               decattn_bf16* out, float* lse, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return gqa_decode_dv(q, k, v, kv, seqlens, max_seqlen, b, s, hq, hkv, d, d, scale, out, lse, workspace,
                       workspace_bytes, stream);
}

// ------------------------------------------------------------------ MLA

static int check_proj(const void* a, const void* w, const void* c, int b, int s, int h, int kin, int nout) {
  if (b < 0 || s < 1 || s > kMaxS || h < 1 || kin < 8 || nout < 8) return DECATTN_ERR_INVALID_ARG;
  if (!a || !w || !c) return DECATTN_ERR_INVALID_ARG;
  if (kin % 8 || nout % 8) return DECATTN_ERR_UNSUPPORTED;
  if (!aligned16(a) || !aligned16(w) || !aligned16(c)) return DECATTN_ERR_INVALID_ARG;
  if (h > 65535 || (long long)b * s > 65535LL * 64) return DECATTN_ERR_INVALID_ARG;
  return DECATTN_OK;
}

int mla_absorb_q(const decattn_bf16* q_nope, const decattn_bf16* w_uk, decattn_bf16* qz, const int32_t* seqlens,
                 int b, int s, int h, int d, int k, float scale, cudaStream_t stream) {
  if (int rc = check_proj(q_nope, w_uk, qz, b, s, h, d, k)) return rc;
  if (b == 0) return DECATTN_OK;
  DeviceState* st = nullptr;
  if (int rc = device_state(&st)) return rc;
  ProjLaunch a{st->err, wait_limit(), q_nope, w_uk, qz, seqlens, b, s, h, d, k, scale};
  return launch_proj(a, st->sms, stream) == cudaSuccess ? DECATTN_OK : DECATTN_ERR_CUDA;
}

int mla_out_proj(const decattn_bf16* o_lat, const decattn_bf16* w_uv, decattn_bf16* out, const int32_t* seqlens,
                 int b, int s, int h, int k, int d, float scale, cudaStream_t stream) {
  if (int rc = check_proj(o_lat, w_uv, out, b, s, h, k, d)) return rc;
  if (b == 0) return DECATTN_OK;
  DeviceState* st = nullptr;
  if (int rc = device_state(&st)) return rc;
  ProjLaunch a{st->err, wait_limit(), o_lat, w_uv, out, seqlens, b, s, h, k, d, scale};
  return launch_proj(a, st->sms, stream) == cudaSuccess ? DECATTN_OK : DECATTN_ERR_CUDA;
}

int mla_decompress_kv(const decattn_bf16* z, const decattn_bf16* k_pe, const decattn_bf16* w_uk,
                      const decattn_bf16* w_uv, int rows, int h, int d, int k, int p, decattn_bf16* k_out,
                      decattn_bf16* v_out, cudaStream_t stream) {
  if (rows < 0 || h < 1 || d < 1 || k < 1 || p < 0) return DECATTN_ERR_INVALID_ARG;
  if (rows == 0) return DECATTN_OK;
  if (!z || !k_pe || !w_uk || !w_uv || !k_out || !v_out) return DECATTN_ERR_INVALID_ARG;
  if (!mla_expand_supported(d, k, p)) return DECATTN_ERR_UNSUPPORTED;
  if (!aligned16(z) || !aligned16(k_pe) || !aligned16(w_uk) || !aligned16(w_uv) || !aligned16(k_out) ||
      !aligned16(v_out))
    return DECATTN_ERR_INVALID_ARG;
  if (h > 65535 * 8 || (long long)h * k > INT_MAX) return DECATTN_ERR_INVALID_ARG;
  DeviceState* st = nullptr;
  if (int rc = device_state(&st)) return rc;
  ExpandLaunch a{z, k_pe, w_uk, w_uv, k_out, v_out, rows, h, k, st->err, wait_limit()};
  return launch_mla_expand(a, stream) == cudaSuccess ? DECATTN_OK : DECATTN_ERR_CUDA;
}

int attn_merge_lse(const decattn_bf16* out_a, const float* lse_a, const decattn_bf16* out_b, const float* lse_b,
                   int rows, int d, decattn_bf16* out, float* lse, cudaStream_t stream) {
  if (rows < 0 || d < 8 || d % 8) return DECATTN_ERR_INVALID_ARG;
  if (rows == 0) return DECATTN_OK;
  if (!out_a || !lse_a || !out_b || !lse_b || !out) return DECATTN_ERR_INVALID_ARG;
  if (!aligned16(out_a) || !aligned16(out_b) || !aligned16(out)) return DECATTN_ERR_INVALID_ARG;
  if ((long long)rows * (d / 8) > (long long)INT_MAX * 256) return DECATTN_ERR_INVALID_ARG;
  DeviceState* st = nullptr;
  if (int rc = device_state(&st)) return rc;
  return launch_merge2(out_a, lse_a, out_b, lse_b, rows, d, out, lse, stream) == cudaSuccess ? DECATTN_OK
                                                                                               : DECATTN_ERR_CUDA;
}

size_t mla_decode_workspace_size(int b, int s, int h, int k, int max_seqlen) {
  if (b < 1 || s < 1 || h < 1 || k < 1) return 0;
  DeviceState* st = nullptr;
  if (device_state(&st)) return 0;
  const Plan pl = mla_plan(b, s, h, k, max_seqlen, st->sms);
  const MlaTail tail = mla_tail(b, s, h, max_seqlen, st->sms, pl);
  if (tail.k > 0) return mla_tail_bytes(tail, k);
  return partial_bytes((long long)b * h * s, pl.nsplit, k, kMlaPartialBytes);
}

int mla_decode(const decattn_bf16* qz, const decattn_bf16* q_pe, const decattn_bf16* z, const decattn_bf16* k_pe,
               decattn_kv kv, const int32_t* seqlens, int max_seqlen, int b, int s, int h, int k, int p,
               float scale, decattn_bf16* o_lat, float* lse, void* workspace, size_t workspace_bytes,
               cudaStream_t stream) {
  if (b < 0 || s < 1 || s > kMaxS || h < 1 || max_seqlen < 0) return DECATTN_ERR_INVALID_ARG;
  if (b == 0) return DECATTN_OK;
  if (!qz || !q_pe || !z || !k_pe || !seqlens || !o_lat) return DECATTN_ERR_INVALID_ARG;
  if (!mla_supported(k, p)) return DECATTN_ERR_UNSUPPORTED;
  if (!aligned16(qz) || !aligned16(q_pe) || !aligned16(z) || !aligned16(k_pe) || !aligned16(o_lat))
    return DECATTN_ERR_INVALID_ARG;
  if (b > 65535 || (long long)b * h * s > INT_MAX / 2) return DECATTN_ERR_INVALID_ARG;
  if (int rc = check_kv(kv, b, max_seqlen)) return rc;
  DeviceState* st = nullptr;
  if (int rc = device_state(&st)) return rc;
  const Plan pl = mla_plan(b, s, h, k, max_seqlen, st->sms);
  const long long rows = (long long)b * h * s;
  const MlaTail tail = mla_tail(b, s, h, max_seqlen, st->sms, pl);
  const size_t need = tail.k > 0 ? mla_tail_bytes(tail, k) : partial_bytes(rows, pl.nsplit, k, kMlaPartialBytes);
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace))) return DECATTN_ERR_WORKSPACE;
  MlaLaunch a;
  a.qz = qz;
  a.q_pe = q_pe;
  a.z = z;
  a.k_pe = k_pe;
  a.seqlens = seqlens;
  a.block_table = kv.block_table;
  a.max_pages = kv.max_pages;
  a.paged = kv.paged;
  a.capacity = kv.capacity;
  a.num_pages = kv.num_pages;
  a.b = b;
  a.s = s;
  a.h = h;
  a.k = k;
  a.p = p;
  a.nsplit = pl.nsplit;
  a.chunk = pl.chunk;
  a.scale = scale;
  a.o_lat = o_lat;
  a.lse = lse;
  a.ws_o = pl.nsplit > 1 ? workspace : nullptr;
  a.ws_lse = pl.nsplit > 1 ? reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                                       align256((size_t)rows * pl.nsplit * k * kMlaPartialBytes))
                           : nullptr;
  a.tail_whole = tail.whole;
  a.tail_units = tail.units;
  a.tail_k = tail.k;
  a.tail_chunk = tail.chunk;
  if (tail.k > 0) {
    const size_t trows = (size_t)tail.units * 128 * tail.k;
    a.ws_o = workspace;
    a.ws_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) + align256(trows * k * kMlaPartialBytes));
  }
  a.err = st->err;
  a.wait_ns = wait_limit();
  a.test_timeout = g_test_timeout.load();
  g_last_splits.store(tail.k > 0 ? tail.k : pl.nsplit);  // the tail units' chunk count
  if (launch_mla_latent(a, stream) != cudaSuccess) return DECATTN_ERR_CUDA;
  if (tail.k > 0) {
    if (launch_combine_tail(a.ws_o, a.ws_lse, seqlens, tail.units, tail.whole, (int)ceil_div((long long)h * s, 128),
                            h * s, tail.k, tail.chunk, k, o_lat, lse, stream) != cudaSuccess)
      return DECATTN_ERR_CUDA;
  } else if (pl.nsplit > 1) {
    if (launch_combine(a.ws_o, true, a.ws_lse, seqlens, (int)rows, h * s, pl.nsplit, pl.chunk, k, o_lat, lse, stream) !=
        cudaSuccess)
      return DECATTN_ERR_CUDA;
  }
  return DECATTN_OK;
}

}  // extern "C"
