// api.cu -- C ABI: argument checks, workspace layout and launches.
//
// The checks restate the load-time checks of the load.rs source page
// (hidden % 256 == 0; expert width a multiple of the 64-code group;
// top_k * rows < SLOT_STRIDE; shared expert width == expert width; Q4 code
// offsets 16-byte aligned, kept here as 256-byte alignment of every tensor)
// plus the limits of these kernels.
#include <cuda.h>

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "decode.cuh"
#include "moe_api.h"
#include "prefill.cuh"

static_assert(MOE_PREFILL_KERNELS == moe::kPfStages, "prefill kernel count");

namespace {

thread_local std::string g_err;

int fail(int code, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

size_t align256(size_t n) { return (n + 255) & ~(size_t)255; }

struct WsLayout {
  size_t cnt, lgw, lgp, xbuf, hfrag, ypart, total;
};

WsLayout ws_layout(int H, int I, int nl, int nb) {
  WsLayout w{};
  size_t off = 0;
  w.cnt = off;
  off += align256((size_t)nl * moe::kCntPerLayer * 4);
  w.lgw = off;
  off += align256((size_t)2 * moe::kMaxGrid * moe::kLogitWords * 8);
  w.lgp = off;
  off += align256((size_t)2 * moe::kMaxGrid * moe::kLogitWords * 8);
  w.xbuf = off;
  off += align256((size_t)nl * nb * H * 4);
  w.hfrag = off;
  off += align256((size_t)64 * I * 16);
  w.ypart = off;
  off += align256((size_t)64 * nb * H * 4);
  w.total = off;
  return w;
}

// Bytes from a record's base to the end of its last tensor (codes, scales
// and biases of gate_up and down at width `bits`).
uint32_t record_span(const moe_q &gu, const moe_q &dn, int I, int H, int bits) {
  const uint64_t gc = (uint64_t)2 * I * H * bits / 8, gs = (uint64_t)2 * I * (H / 64) * 2;
  const uint64_t dc = (uint64_t)H * I * bits / 8, ds = (uint64_t)H * (I / 64) * 2;
  uint64_t e = gu.w + gc;
  e = e > gu.s + gs ? e : gu.s + gs;
  e = e > gu.b + gs ? e : gu.b + gs;
  e = e > dn.w + dc ? e : dn.w + dc;
  e = e > dn.s + ds ? e : dn.s + ds;
  e = e > dn.b + ds ? e : dn.b + ds;
  return (uint32_t)((e + 15) & ~(uint64_t)15);
}

int check_q(const moe_q &q, uint32_t out, uint32_t inp, const char *what, int l) {
  if (q.out != out || q.inp != inp)
    return fail(MOE_ESHAPE, "layer %d %s: shape [%u][%u], expected [%u][%u]", l, what, q.out, q.inp, out, inp);
  if ((q.w | q.s | q.b) & 255u) return fail(MOE_EALIGN, "layer %d %s: offsets must be 256-byte aligned", l, what);
  return MOE_OK;
}

int check_layers(const moe_layer *layers, int nl, int nb) {
  if (!layers) return fail(MOE_EINVAL, "layers is NULL");
  if (nl < 1 || nl > MOE_MAX_LAYERS) return fail(MOE_EINVAL, "n_layers %d outside 1..%d", nl, MOE_MAX_LAYERS);
  if (nb < 1 || nb > MOE_MAX_NB) return fail(MOE_EINVAL, "nb %d outside 1..%d", nb, MOE_MAX_NB);
  const moe_layer &L0 = layers[0];
  const uint32_t H = L0.hidden, E = L0.n_experts, K = L0.top_k, I = L0.inter, bits = L0.bits;
  const bool mixed = L0.expert_bits != nullptr;
  if (H == 0 || H % 256) return fail(MOE_ESHAPE, "hidden %u must be a positive multiple of 256", H);
  if (H > 2048) return fail(MOE_ESHAPE, "hidden %u above the decode kernel's limit 2048", H);
  if (I == 0 || I % 128) return fail(MOE_ESHAPE, "inter %u must be a positive multiple of 128", I);
  if (I > 1024) return fail(MOE_ESHAPE, "inter %u above the decode kernel's limit 1024", I);
  if (E < 1 || E > 1024) return fail(MOE_ESHAPE, "n_experts %u outside 1..1024", E);
  if (K < 1 || K > E || K > 32) return fail(MOE_ESHAPE, "top_k %u outside 1..min(n_experts, 32)", K);
  if (K * (uint32_t)nb >= MOE_SLOT_STRIDE) return fail(MOE_ESHAPE, "top_k * nb = %u must be < 64", K * nb);
  if (!mixed && bits != 2 && bits != 3 && bits != 4) return fail(MOE_ESHAPE, "bits %u not in {2,3,4}", bits);
  for (int l = 0; l < nl; l++) {
    const moe_layer &L = layers[l];
    if (L.hidden != H || L.n_experts != E || L.top_k != K || L.inter != I)
      return fail(MOE_ESHAPE, "layer %d: dimensions differ from layer 0", l);
    if ((L.expert_bits != nullptr) != mixed)
      return fail(MOE_EINVAL, "layer %d: expert_bits must be set on every layer or on none", l);
    if (!mixed && L.bits != bits) return fail(MOE_ESHAPE, "layer %d: bits differ from layer 0", l);
    if (!(L.cut_weak >= 0.f && L.cut_weak <= 1.f))
      return fail(MOE_EINVAL, "layer %d: cut_weak %g outside [0, 1]", l, (double)L.cut_weak);
    if (L.group != 64) return fail(MOE_ESHAPE, "layer %d: group %u, only 64 is supported", l, L.group);
    if (L.flags & ~(uint32_t)(MOE_RESIDUAL | MOE_PRENORM | MOE_LOOKAHEAD | MOE_TEST_WITHHOLD))
      return fail(MOE_EINVAL, "layer %d: unknown flags 0x%x", l, L.flags);
    if (!L.router || !L.expert_addr) return fail(MOE_EINVAL, "layer %d: router / expert_addr NULL", l);
    if ((uintptr_t)L.router & 15u) return fail(MOE_EALIGN, "layer %d: router not 16-byte aligned", l);
    if (!L.shared_gate != !L.shared_record)
      return fail(MOE_EINVAL, "layer %d: shared_gate and shared_record must both be set or both NULL", l);
    if (L.shared_gate) {
      if (((uintptr_t)L.shared_gate | (uintptr_t)L.shared_record) & 15u)
        return fail(MOE_EALIGN, "layer %d: shared gate / record not 16-byte aligned", l);
      int r;
      if ((r = check_q(L.sh_gate_up, 2 * I, H, "sh_gate_up", l))) return r;
      if ((r = check_q(L.sh_down, H, I, "sh_down", l))) return r;
    }
    int r;
    if (mixed) {
      for (int i = 0; i < 3; i++) {
        if ((r = check_q(L.gate_up_w[i], 2 * I, H, "gate_up_w", l))) return r;
        if ((r = check_q(L.down_w[i], H, I, "down_w", l))) return r;
      }
    } else {
      if ((r = check_q(L.gate_up, 2 * I, H, "gate_up", l))) return r;
      if ((r = check_q(L.down, H, I, "down", l))) return r;
    }
  }
  return MOE_OK;
}

unsigned long long timeout_ns() {
  const char *s = getenv("MOE_TIMEOUT_MS");
  double ms = s ? atof(s) : 1000.0;
  if (!(ms > 0)) ms = 1000.0;
  return (unsigned long long)(ms * 1e6);
}

bool overlap(const void *a, size_t na, const void *b, size_t nb) {
  const char *pa = (const char *)a, *pb = (const char *)b;
  return pa < pb + nb && pb < pa + na;
}

int run(const moe_layer *layers, int nl, const float *x, int nb, float *out, void *work, size_t work_bytes,
        uint64_t *slot_tab, float *wmap, uint32_t *topk_idx, float *topk_w, float *logits, int *status,
        moe_stream_t stream, int route_only, uint64_t *trace = nullptr) {
  const moe_layer &L0 = layers[0];
  const int H = (int)L0.hidden, E = (int)L0.n_experts, I = (int)L0.inter;
  if (!x) return fail(MOE_EINVAL, "x is NULL");
  if (!route_only && !out) return fail(MOE_EINVAL, "out is NULL");
  if (!status) return fail(MOE_EINVAL, "dev_status is NULL");
  if (!work) return fail(MOE_EINVAL, "work is NULL");
  if ((uintptr_t)work & 255u) return fail(MOE_EALIGN, "work must be 256-byte aligned");
  if (!route_only && overlap(x, (size_t)nb * H * 4, out, (size_t)nb * H * 4))
    return fail(MOE_EINVAL, "out overlaps x");
  const WsLayout w = ws_layout(H, I, nl, nb);
  if (work_bytes < w.total) return fail(MOE_ENOSPACE, "work holds %zu bytes, %zu needed", work_bytes, w.total);

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(MOE_ECUDA, "cudaGetDevice failed");

  static_assert(sizeof(moe::FwdParams) < 32000, "kernel parameters too large");
  moe::FwdParams p;
  memset(&p, 0, sizeof p);
  p.H = H, p.E = E, p.K = (int)L0.top_k, p.I = I, p.nb = nb, p.nl = nl;
  p.bits = L0.expert_bits ? 0 : (int)L0.bits;  // 0: the mixed-width kernel instance
  p.route_only = route_only;
  p.x = x, p.out = out;
  p.slot_tab = slot_tab, p.wmap = wmap, p.topk_idx = topk_idx, p.topk_w = topk_w, p.logits_out = logits;
  p.status = status;
  char *base = (char *)work;
  p.cnt = (unsigned *)(base + w.cnt);
  p.lgw = (unsigned long long *)(base + w.lgw);
  p.lgp = (unsigned long long *)(base + w.lgp);
  p.xbuf = (float *)(base + w.xbuf);
  p.hfrag = (uint16_t *)(base + w.hfrag);
  p.ypart = (float *)(base + w.ypart);
  p.timeout_ns = timeout_ns();
  p.trace = reinterpret_cast<unsigned long long *>(trace);
  for (int l = 0; l < nl; l++) {
    const moe_layer &L = layers[l];
    moe::LayerP &q = p.L[l];
    q.router = L.router;
    q.sgate = L.shared_gate;
    q.srec = (const uint8_t *)L.shared_record;
    q.eaddr = L.expert_addr;
    q.gu = {(uint32_t)L.gate_up.w, (uint32_t)L.gate_up.s, (uint32_t)L.gate_up.b};
    q.dn = {(uint32_t)L.down.w, (uint32_t)L.down.s, (uint32_t)L.down.b};
    q.sgu = {(uint32_t)L.sh_gate_up.w, (uint32_t)L.sh_gate_up.s, (uint32_t)L.sh_gate_up.b};
    q.sdn = {(uint32_t)L.sh_down.w, (uint32_t)L.sh_down.s, (uint32_t)L.sh_down.b};
    q.flags = L.flags & (MOE_RESIDUAL | MOE_PRENORM | MOE_LOOKAHEAD);
    if (L.flags & MOE_TEST_WITHHOLD) p.withhold = 1;
    if ((L.flags & MOE_LOOKAHEAD) && l > 0) p.lookahead = 1;
    q.ebits = L.expert_bits;
    q.etier = L.expert_tier;
    q.cut_w = L.cut_weak;
    q.la_idx = L.lookahead_idx;
    q.span = record_span(L.gate_up, L.down, I, H, L.bits);
    for (int i = 0; i < 3; i++) q.span_w[i] = record_span(L.gate_up_w[i], L.down_w[i], I, H, 4 - i);
    if (L.expert_bits)
      for (int i = 0; i < 3; i++) {
        q.guw[i] = {(uint32_t)L.gate_up_w[i].w, (uint32_t)L.gate_up_w[i].s, (uint32_t)L.gate_up_w[i].b};
        q.dnw[i] = {(uint32_t)L.down_w[i].w, (uint32_t)L.down_w[i].s, (uint32_t)L.down_w[i].b};
      }
  }
  int grid = 0, smem = 0;
  if (moe::decode_plan(dev, p, &grid, &smem) != 0)
    return fail(MOE_ECUDA, "decode kernel cannot be resident on this device (hidden %d, experts %d)", H, E);
  cudaStream_t st = (cudaStream_t)stream;
  // counters and the logit exchange words (adjacent) and the status start at
  // zero every call: a small kernel clears them, the decode kernel follows it
  cudaError_t e = moe::launch_decode(p, grid, smem, st, (size_t)(w.xbuf - w.cnt));
  if (e != cudaSuccess) return fail(MOE_ECUDA, "launch failed: %s", cudaGetErrorString(e));
  return MOE_OK;
}

int check_offsets_fit(const moe_layer *layers, int nl) {
  for (int l = 0; l < nl; l++) {
    const moe_layer &L = layers[l];
    const moe_q *qs[10] = {&L.gate_up,      &L.down,         &L.sh_gate_up,   &L.sh_down,      &L.gate_up_w[0],
                           &L.gate_up_w[1], &L.gate_up_w[2], &L.down_w[0],    &L.down_w[1],    &L.down_w[2]};
    for (const moe_q *q : qs)
      if ((q->w | q->s | q->b) >> 32) return fail(MOE_ESHAPE, "layer %d: record offsets must be < 4 GiB", l);
  }
  return MOE_OK;
}

// ---- fixed scratch for callers that cannot allocate device memory
//
// Some callers cannot make device allocations at the point where they run
// the MoE step: code being recorded into a CUDA graph (an allocation there
// is either forbidden or turns into a graph node the caller did not plan),
// engines that hand every byte of device memory to their own pool and allow
// no outside allocations, and latency-critical loops that must not risk the
// implicit device synchronisation a cudaMalloc / cudaFree may cause.  For
// them moe_forward_noalloc runs the same kernel on this fixed array instead
// of a caller-provided workspace.  The array lives for the life of the
// process on every GPU that loads this library.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MOE_NOALLOC_MAX_WORKSPACE];

std::mutex g_noalloc_mu;

// The array's device address depends on the CUDA context that loaded this
// library's module, not only on the device number: after cudaDeviceReset, or
// with another context current on the same device, an address looked up
// earlier is no longer valid.  So the cache is keyed by the driver's context
// id (unique for the life of the process; a context made after a reset gets
// a new id).  The two driver calls are reached through the runtime's entry
// point table, so the library needs no link against libcuda.
struct NoallocEntry {
  unsigned long long ctx_id;
  void *ptr;
};
constexpr int kNoallocCache = 64;
NoallocEntry g_noalloc_cache[kNoallocCache];
int g_noalloc_used = 0;

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

// Id of the context current on this thread (0 if none is current yet).
int current_ctx_id(unsigned long long *id) {
  static CtxGetCurrentFn get_cur = nullptr;
  static CtxGetIdFn get_id = nullptr;
  if (!get_cur || !get_id) {
    cudaDriverEntryPointQueryResult q1 = cudaDriverEntryPointSymbolNotFound, q2 = q1;
    void *f1 = nullptr, *f2 = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 4000, cudaEnableDefault, &q1) != cudaSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) != cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess || q2 != cudaDriverEntryPointSuccess || !f1 || !f2)
      return fail(MOE_ECUDA, "driver entry points cuCtxGetCurrent / cuCtxGetId are unavailable");
    get_cur = reinterpret_cast<CtxGetCurrentFn>(f1);
    get_id = reinterpret_cast<CtxGetIdFn>(f2);
  }
  CUcontext ctx = nullptr;
  if (get_cur(&ctx) != CUDA_SUCCESS) return fail(MOE_ECUDA, "cuCtxGetCurrent failed");
  *id = 0;
  if (ctx && get_id(ctx, id) != CUDA_SUCCESS) return fail(MOE_ECUDA, "cuCtxGetId failed");
  return MOE_OK;
}

// Device address of the scratch array in the current context: looked up once
// per context with cudaGetSymbolAddress (which also makes the runtime's
// context current if none was), then served from the cache.
int noalloc_scratch(void **out) {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  unsigned long long id = 0;
  int r = current_ctx_id(&id);
  if (r != MOE_OK) return r;
  for (int i = 0; id != 0 && i < g_noalloc_used; i++)
    if (g_noalloc_cache[i].ctx_id == id) {
      *out = g_noalloc_cache[i].ptr;
      return MOE_OK;
    }
  void *p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess || !p)
    return fail(MOE_ECUDA, "cudaGetSymbolAddress of the fixed scratch failed: %s", cudaGetErrorString(e));
  if (id == 0 && (r = current_ctx_id(&id)) != MOE_OK) return r;
  if (id != 0) {
    // a full table recycles its oldest entry (contexts of long-gone resets)
    const int slot = g_noalloc_used < kNoallocCache ? g_noalloc_used++ : (int)(id % kNoallocCache);
    g_noalloc_cache[slot] = {id, p};
  }
  *out = p;
  return MOE_OK;
}

// ---- prefill chunk

constexpr int kMaxPrefillRows = 1 << 20;

int check_prefill(const moe_layer *L, int t) {
  if (!L) return fail(MOE_EINVAL, "layer is NULL");
  if (t < 1 || t > kMaxPrefillRows) return fail(MOE_EINVAL, "t %d outside 1..%d", t, kMaxPrefillRows);
  const uint32_t H = L->hidden, E = L->n_experts, K = L->top_k, I = L->inter;
  if (H == 0 || H % 256) return fail(MOE_ESHAPE, "hidden %u must be a positive multiple of 256", H);
  if (H > 16384) return fail(MOE_ESHAPE, "hidden %u above 16384", H);
  if (I == 0 || I % 64 || I > 16384) return fail(MOE_ESHAPE, "inter %u must be a multiple of 64 in 64..16384", I);
  if (E < 1 || E > 1024) return fail(MOE_ESHAPE, "n_experts %u outside 1..1024", E);
  if (K < 1 || K > E || K > 32) return fail(MOE_ESHAPE, "top_k %u outside 1..min(n_experts, 32)", K);
  // the GEMMs reach a row of the grouped operands (x^ rows, h), stored as
  // k-panels of t * (top_k + 1) rows, with a signed 32-bit tensor-map
  // coordinate: panel * t * (top_k + 1) + row
  const uint64_t ent = (uint64_t)t * (K + 1);
  if ((uint64_t)(H / 64) * ent > (uint64_t)INT32_MAX || (uint64_t)(I / 64) * ent > (uint64_t)INT32_MAX)
    return fail(MOE_ESHAPE, "t %d x (top_k + 1) rows in %u k-panels exceed the 2^31 rows a tensor-map coordinate reaches",
                t, (H > I ? H : I) / 64);
  if (L->expert_bits) return fail(MOE_EINVAL, "mixed record widths (expert_bits) are supported by decode only");
  if (L->expert_tier || L->cut_weak != 0.f)
    return fail(MOE_EINVAL, "host-memory records (expert_tier, cut_weak) are supported by decode only");
  if (L->bits != 2 && L->bits != 3 && L->bits != 4) return fail(MOE_ESHAPE, "bits %u not in {2,3,4}", L->bits);
  // the GEMMs stage code rows with 16-byte copies: a 3-bit row (3 * in / 8
  // bytes) is 16-byte aligned when in is a multiple of 128
  if (L->bits == 3 && I % 128)
    return fail(MOE_ESHAPE, "3-bit prefill needs inter %% 128 == 0 (16-byte code rows); inter %u", I);
  if (L->group != 64) return fail(MOE_ESHAPE, "group %u, only 64 is supported", L->group);
  if (L->flags & ~(uint32_t)(MOE_RESIDUAL | MOE_PRENORM | MOE_LOOKAHEAD | MOE_TEST_WITHHOLD))
    return fail(MOE_EINVAL, "unknown flags 0x%x", L->flags);
  if (!L->router || !L->expert_addr) return fail(MOE_EINVAL, "router / expert_addr NULL");
  if ((uintptr_t)L->router & 15u) return fail(MOE_EALIGN, "router not 16-byte aligned");
  if (!L->shared_gate != !L->shared_record)
    return fail(MOE_EINVAL, "shared_gate and shared_record must both be set or both NULL");
  int r;
  if (L->shared_gate) {
    if (((uintptr_t)L->shared_gate | (uintptr_t)L->shared_record) & 15u)
      return fail(MOE_EALIGN, "shared gate / record not 16-byte aligned");
    if ((r = check_q(L->sh_gate_up, 2 * I, H, "sh_gate_up", 0))) return r;
    if ((r = check_q(L->sh_down, H, I, "sh_down", 0))) return r;
  }
  if ((r = check_q(L->gate_up, 2 * I, H, "gate_up", 0))) return r;
  if ((r = check_q(L->down, H, I, "down", 0))) return r;
  return check_offsets_fit(L, 1);
}

size_t prefill_bytes(const moe_layer *L, int t) {
  return moe::pf_workspace_bytes((int)L->hidden, (int)L->n_experts, (int)L->top_k, (int)L->inter, t);
}

int run_prefill(const moe_layer *L, const float *x, int t, uint16_t *out, void *work, size_t work_bytes,
                uint32_t *topk_idx, float *topk_w, int *status, moe_stream_t stream, int route_only,
                void *const *events = nullptr) {
  const int H = (int)L->hidden;
  if (!x) return fail(MOE_EINVAL, "x is NULL");
  if (!route_only && !out) return fail(MOE_EINVAL, "out is NULL");
  if (!status) return fail(MOE_EINVAL, "dev_status is NULL");
  if (!work) return fail(MOE_EINVAL, "work is NULL");
  if ((uintptr_t)work & 255u) return fail(MOE_EALIGN, "work must be 256-byte aligned");
  if ((uintptr_t)x & 15u) return fail(MOE_EALIGN, "x must be 16-byte aligned");
  if (!route_only && overlap(x, (size_t)t * H * 4, out, (size_t)t * H * 2))
    return fail(MOE_EINVAL, "out overlaps x");
  const size_t need = prefill_bytes(L, t);
  if (work_bytes < need) return fail(MOE_ENOSPACE, "work holds %zu bytes, %zu needed", work_bytes, need);
  moe::PfParams p;
  memset(&p, 0, sizeof p);
  p.H = H, p.E = (int)L->n_experts, p.K = (int)L->top_k, p.I = (int)L->inter, p.t = t;
  p.bits = (int)L->bits;
  p.flags = L->flags & (MOE_RESIDUAL | MOE_PRENORM);
  p.withhold = (L->flags & MOE_TEST_WITHHOLD) != 0;
  p.route_only = route_only;
  p.x = x, p.out = out;
  p.router = L->router, p.sgate = L->shared_gate;
  p.srec = (const uint8_t *)L->shared_record;
  p.eaddr = L->expert_addr;
  p.gu = {(uint32_t)L->gate_up.w, (uint32_t)L->gate_up.s, (uint32_t)L->gate_up.b};
  p.dn = {(uint32_t)L->down.w, (uint32_t)L->down.s, (uint32_t)L->down.b};
  p.sgu = {(uint32_t)L->sh_gate_up.w, (uint32_t)L->sh_gate_up.s, (uint32_t)L->sh_gate_up.b};
  p.sdn = {(uint32_t)L->sh_down.w, (uint32_t)L->sh_down.s, (uint32_t)L->sh_down.b};
  p.topk_out = topk_idx, p.topkw_out = topk_w;
  p.status = status;
  p.timeout_ns = timeout_ns();
  moe::pf_carve(p, work);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&p.n_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return fail(MOE_ECUDA, "device query failed");
  const char *why = "";
  if (moe::pf_tensor_maps(p, &why) != 0) return fail(MOE_ECUDA, "%s", why);
  const cudaError_t e = moe::pf_launch(p, (cudaStream_t)stream, reinterpret_cast<cudaEvent_t const *>(events));
  if (e != cudaSuccess) return fail(MOE_ECUDA, "prefill launch failed: %s", cudaGetErrorString(e));
  return MOE_OK;
}

}  // namespace

extern "C" {

const char *moe_last_error(void) { return g_err.c_str(); }

size_t moe_forward_workspace(const moe_layer *layers, int n_layers, int nb) {
  if (check_layers(layers, n_layers, nb) != MOE_OK) return 0;
  const moe_layer &L0 = layers[0];
  return ws_layout((int)L0.hidden, (int)L0.inter, n_layers, nb).total;
}

int moe_forward(const moe_layer *layers, int n_layers, const float *x, int nb, float *out, void *work,
                size_t work_bytes, uint64_t *slot_tab, float *wmap, uint32_t *topk_idx, int *dev_status,
                moe_stream_t stream) {
  int r = check_layers(layers, n_layers, nb);
  if (r == MOE_OK) r = check_offsets_fit(layers, n_layers);
  if (r != MOE_OK) return r;
  return run(layers, n_layers, x, nb, out, work, work_bytes, slot_tab, wmap, topk_idx, nullptr, nullptr,
             dev_status, stream, 0);
}

int moe_forward_traced(const moe_layer *layers, int n_layers, const float *x, int nb, float *out, void *work,
                       size_t work_bytes, uint64_t *slot_tab, float *wmap, uint32_t *topk_idx, int *dev_status,
                       uint64_t *phase_ns, moe_stream_t stream) {
  int r = check_layers(layers, n_layers, nb);
  if (r == MOE_OK) r = check_offsets_fit(layers, n_layers);
  if (r != MOE_OK) return r;
  if (!phase_ns) return fail(MOE_EINVAL, "phase_ns is NULL");
  return run(layers, n_layers, x, nb, out, work, work_bytes, slot_tab, wmap, topk_idx, nullptr, nullptr,
             dev_status, stream, 0, phase_ns);
}

int moe_forward_noalloc(const moe_layer *layers, int n_layers, const float *x, int nb, float *out,
                        uint64_t *slot_tab, float *wmap, uint32_t *topk_idx, int *dev_status,
                        moe_stream_t stream) {
  int r = check_layers(layers, n_layers, nb);
  if (r == MOE_OK) r = check_offsets_fit(layers, n_layers);
  if (r != MOE_OK) return r;
  const moe_layer &L0 = layers[0];
  const size_t need = ws_layout((int)L0.hidden, (int)L0.inter, n_layers, nb).total;
  if (need > MOE_NOALLOC_MAX_WORKSPACE)
    return fail(MOE_ENOSPACE, "these layers need %zu bytes of scratch; the fixed scratch holds %u", need,
                (unsigned)MOE_NOALLOC_MAX_WORKSPACE);
  void *work = nullptr;
  if ((r = noalloc_scratch(&work)) != MOE_OK) return r;
  return run(layers, n_layers, x, nb, out, work, MOE_NOALLOC_MAX_WORKSPACE, slot_tab, wmap, topk_idx, nullptr,
             nullptr, dev_status, stream, 0);
}

int moe_route(const moe_layer *L, const float *x, int nb, float *logits, uint32_t *topk_idx, float *topk_w,
              uint64_t *slot_row, float *wmap_row, void *work, size_t work_bytes, int *dev_status,
              moe_stream_t stream) {
  int r = check_layers(L, 1, nb);
  if (r == MOE_OK) r = check_offsets_fit(L, 1);
  if (r != MOE_OK) return r;
  if (!topk_idx || !topk_w || !slot_row || !wmap_row)
    return fail(MOE_EINVAL, "topk_idx, topk_w, slot_row and wmap_row are required");
  return run(L, 1, x, nb, nullptr, work, work_bytes, slot_row, wmap_row, topk_idx, topk_w, logits, dev_status,
             stream, 1);
}

size_t moe_prefill_workspace(const moe_layer *L, int t) {
  if (check_prefill(L, t) != MOE_OK) return 0;
  return prefill_bytes(L, t);
}

int moe_prefill(const moe_layer *L, const float *x, int t, uint16_t *out, void *work, size_t work_bytes,
                uint32_t *topk_idx, int *dev_status, moe_stream_t stream) {
  const int r = check_prefill(L, t);
  if (r != MOE_OK) return r;
  return run_prefill(L, x, t, out, work, work_bytes, topk_idx, nullptr, dev_status, stream, 0);
}

int moe_prefill_timed(const moe_layer *L, const float *x, int t, uint16_t *out, void *work, size_t work_bytes,
                      uint32_t *topk_idx, int *dev_status, void *const *events, moe_stream_t stream) {
  const int r = check_prefill(L, t);
  if (r != MOE_OK) return r;
  if (!events) return fail(MOE_EINVAL, "events is NULL");
  for (int i = 0; i <= MOE_PREFILL_KERNELS; i++)
    if (!events[i]) return fail(MOE_EINVAL, "events[%d] is NULL", i);
  return run_prefill(L, x, t, out, work, work_bytes, topk_idx, nullptr, dev_status, stream, 0, events);
}

int moe_prefill_group(const moe_layer *L, const float *x, int t, uint32_t *topk_idx, float *topk_w,
                      int32_t *group_offs, int32_t *group_rows, float *group_w, void *work, size_t work_bytes,
                      int *dev_status, moe_stream_t stream) {
  int r = check_prefill(L, t);
  if (r != MOE_OK) return r;
  if (!topk_idx || !topk_w || !group_offs || !group_rows || !group_w)
    return fail(MOE_EINVAL, "topk_idx, topk_w, group_offs, group_rows and group_w are required");
  if ((r = run_prefill(L, x, t, nullptr, work, work_bytes, topk_idx, topk_w, dev_status, stream, 1))) return r;
  moe::PfParams p;
  memset(&p, 0, sizeof p);
  p.H = (int)L->hidden, p.E = (int)L->n_experts, p.K = (int)L->top_k, p.I = (int)L->inter, p.t = t;
  moe::pf_carve(p, work);
  const int G = p.E + (L->shared_gate ? 1 : 0);
  const size_t ent = (size_t)t * p.K + (L->shared_gate ? (size_t)t : 0);
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(group_offs, p.offs, (size_t)(G + 1) * 4, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(group_rows, p.rows, ent * 4, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(group_w, p.wts, ent * 4, cudaMemcpyDeviceToDevice, st);
  if (e != cudaSuccess) return fail(MOE_ECUDA, "copy of the grouping failed: %s", cudaGetErrorString(e));
  return MOE_OK;
}

}  // extern "C"
