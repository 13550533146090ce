// prefill.cu -- prefill chunk through one MoE layer on the 5th-gen tensor cores.
//
// Steps (the prefill MoE of the struct Gpu page, `pf_experts`: shared expert
// over all rows, routed experts with their rows gathered, computed and
// scatter-added; `ExpertJob` / `prepare_expert_jobs`: rows grouped by expert):
//   prep    x^ (optional unit RMSNorm), its bf16 hi/lo split for the router,
//           its bf16 rounding (k permuted) for the experts, the shared gate
//   router  logits = R [x^_hi | x^_lo] on tcgen05 (R bf16 exact, fp32 TMEM)
//   top-k   per token, softmax over the k chosen; per-(chunk, expert) counts
//   group   scan -> offsets of the groups (experts, then the shared expert
//           with all t tokens) and of their kPfTileN-token chunks; per-chunk
//           bases
//   fill    token lists in ascending token order (stable), routing weights;
//           the tile work lists
//   gate_up per (group, 64 gate + 64 up rows, <= kPfTileN tokens): weights
//           dequantized to bf16 into tensor memory (A), token rows in group
//           order through TMA (B), tcgen05 MMA into TMEM; epilogue
//           h = silu(gate) * up -> bf16
//   down    per (group, 128 output rows, <= kPfTileN tokens): A = dequantized
//           down rows, B = h; epilogue Y[token] += weight * y (fp32)
//   final   out = bf16(Y) (+ x for a residual layer)
// The k order inside every 8-element block is permuted the same way on both
// expert operands so that one mask / FMA pair turns two codes into a bf16
// pair (nibbles j and j+4 of a code word share a register).
#include <cuda_runtime.h>

#include "codec.cuh"
#include "prefill.cuh"
#include "tc05.cuh"

namespace moe {
namespace {

constexpr unsigned FULLM = 0xffffffffu;
constexpr uint32_t kResidualF = 1, kPrenormF = 2;
enum { MODE_ROUTER = 0, MODE_GATE_UP = 1, MODE_DOWN = 2 };


// bf16 bits of f, rounded to nearest even: the hardware conversion (one
// instruction, off the integer pipe the dequant warps lean on)
__device__ __forceinline__ uint32_t f2bf_rn(float f) {
  uint16_t h;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(f));
  return h;
}

// Programmatic dependent launch: every kernel of the chain lets the next one
// launch at once (it then waits, resident, for this grid's completion),
// and waits for the previous kernel's completion and memory before it
// reads that kernel's results.  The next grid launches only when every
// block of this one has started, so a waiting grid never holds resources
// this one still needs.
__device__ __forceinline__ void pdl_launch_next() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait_prev() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_begin() {
  pdl_launch_next();
  pdl_wait_prev();
}

// position of natural index j inside its 8-block under the operand
// permutation: pairs (0,4),(1,5),(2,6),(3,7) are adjacent
__device__ __forceinline__ int perm8(int j) { return (j & 3) * 2 + (j >> 2); }

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(FULLM, v, o);
  return v;
}

// mbar_try_wait, but a thread whose phase is not complete sleeps until it
// completes or about ns nanoseconds pass (instead of a system-set limit)
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

// bounded wait on an mbarrier phase; false (status set) once the limit passes.
// The waiting thread sleeps on the barrier (up to 1 ms a try) rather than
// polling, so the waiting roles leave the issue slots to the dequant warps.
__device__ bool pf_wait(uint64_t *bar, uint32_t par, const PfParams &P) {
  if (mbar_try_wait(bar, par)) return true;
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait_sleep(bar, par, 1000000u)) {
    if (globaltimer() - t0 > P.timeout_ns) {
      atomicCAS(P.status, 0, kStatusTimeout);
      return false;
    }
  }
  return true;
}

// ------------------------------------------------------------ prep
// Block per token, thread per 8-element block: x^, the router operands
// (hi/lo, natural order), the expert operand (bf16 of x^, k permuted within
// the block), the shared gate sigmoid(sg . x^).  16-byte loads and stores.
__global__ void pf_prep(const __grid_constant__ PfParams P) {
  pdl_launch_next();  // (launched after the call's memsets, in plain stream order)
  __shared__ float red[32];
  const int tok = blockIdx.x, H = P.H, nw = blockDim.x >> 5, nb8 = H / 8;
  const float4 *xr = reinterpret_cast<const float4 *>(P.x + (size_t)tok * H);
  float scale = 1.f;
  if (P.flags & kPrenormF) {
    float ss = 0.f;
    for (int b = threadIdx.x; b < nb8; b += blockDim.x) {
      const float4 a = xr[2 * b], c = xr[2 * b + 1];
      ss += a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w + c.x * c.x + c.y * c.y + c.z * c.z + c.w * c.w;
    }
    ss = warp_sum_f(ss);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
    for (int w = 0; w < nw; w++) tot += red[w];
    scale = 1.0f / sqrtf(tot / (float)H + 1e-6f);
    __syncthreads();
  }
  float gdot = 0.f;
  const size_t rb = (size_t)tok * H;
  for (int b = threadIdx.x; b < nb8; b += blockDim.x) {
    const float4 a = xr[2 * b], c = xr[2 * b + 1];
    const float v[8] = {a.x * scale, a.y * scale, a.z * scale, a.w * scale,
                        c.x * scale, c.y * scale, c.z * scale, c.w * scale};
    uint32_t hi[8], lo[8];
#pragma unroll
    for (int j = 0; j < 8; j++) {
      hi[j] = f2bf_rn(v[j]);
      lo[j] = f2bf_rn(v[j] - __uint_as_float(hi[j] << 16));
    }
    *reinterpret_cast<uint4 *>(P.xr_hi + rb + 8 * b) =
        make_uint4(hi[0] | hi[1] << 16, hi[2] | hi[3] << 16, hi[4] | hi[5] << 16, hi[6] | hi[7] << 16);
    *reinterpret_cast<uint4 *>(P.xr_lo + rb + 8 * b) =
        make_uint4(lo[0] | lo[1] << 16, lo[2] | lo[3] << 16, lo[4] | lo[5] << 16, lo[6] | lo[7] << 16);
    // positions 0..7 of the permuted block hold natural indices 0,4,1,5,2,6,3,7
    *reinterpret_cast<uint4 *>(P.xg + rb + 8 * b) =
        make_uint4(hi[0] | hi[4] << 16, hi[1] | hi[5] << 16, hi[2] | hi[6] << 16, hi[3] | hi[7] << 16);
    if (P.sgate) {
      const uint4 g = *reinterpret_cast<const uint4 *>(P.sgate + 8 * b);
      const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
      for (int j = 0; j < 4; j++)
        gdot += __uint_as_float(gw[j] << 16) * v[2 * j] + __uint_as_float(gw[j] & 0xffff0000u) * v[2 * j + 1];
    }
  }
  if (P.sgate) {
    gdot = warp_sum_f(gdot);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = gdot;
    __syncthreads();
    if (threadIdx.x == 0) {
      float tot = 0.f;
      for (int w = 0; w < nw; w++) tot += red[w];
      P.gam[tok] = 1.f / (1.f + expf(-tot));
    }
  }
}

// ------------------------------------------------------------ tensor-core GEMM
//
// Persistent, warp-specialised: one CTA per SM walks tiles blockIdx.x,
// blockIdx.x + gridDim.x, ... of a 128 x N output tile list (N <= 128 for
// the router, <= kPfTileN for the expert GEMMs); K goes in stages of 64.
// B (token rows) passes through a ring of 128B-swizzled shared-memory
// stages (router: six of 128 rows; expert GEMMs: three of up to 320 rows,
// so that a full-width tile takes two k-panels per stage and handshake).
// The expert GEMMs' A (dequantized weight rows) passes through a ring of
// kSA = 3 stages in tensor memory, kPA = 2 k-panels of 32 columns each (row
// r in TMEM lane r, bf16 pairs along k), and feeds tcgen05.mma from there;
// tensor memory holds three such stages beside the two accumulators when a
// tile is at most 160 tokens wide.  The router's A (bf16 rows of R) comes by
// TMA into shared memory beside its B.
//   warp 0      lane 0 issues the tcgen05 MMAs of a stage once its operands
//               have landed and commits them (stage free / accumulator full)
//   warp 1      TMA: B rows (and the router's A rows) of each stage
//   warps 2-9   A producers: all 256 threads stage the codes of four
//               k-panels (128 rows x 128 bytes, plus scale / bias words)
//               into shared memory with coalesced cp.async, three chunks in
//               the air (two for 2- and 3-bit codes); a chunk's two A
//               stages go to the two groups of four warps (w - 2) / 4, and
//               with three stages in the ring a group's next stage was read
//               by the MMAs three stages back, not two:
//               warp w fills rows 32 (w % 4) .. +31 -- the TMEM lanes it may
//               write -- 64 codes a panel, stored as 32 bf16 pairs per panel
//               with tcgen05.st.  Issuing cp.async copies stalls a warp, so
//               the first group issues a chunk's copies after its dequant
//               and the second, which waits longer for its A stage, before
//               that wait.
//   warps 10-13 epilogue: TMEM -> registers -> global, from one of two
//               accumulators while the MMAs fill the other
// Every mbarrier wait is bounded and sleeps on the barrier between tries; a
// wait that gives up records MOE_ETIMEOUT in *status and its role stops, so
// the CTA ends.

constexpr int kWsThreads = 448;
constexpr int kSB = 6;                     // B stages (shared memory), at most
constexpr int kStageRows = 2 * kPfTileN;   // token rows of one expert-GEMM B stage (k-panels of 128 bytes)
constexpr int kSA = 3;                     // A stages (tensor memory; expert GEMMs)
constexpr int kPA = 2;                     // k-panels per A stage (one handshake per two panels)
constexpr int kAccCols = 160;              // TMEM columns of one accumulator (expert GEMMs; N <= 160)
constexpr int kTmemA = 2 * kAccCols;       // first TMEM column of the A ring: kSA x kPA x 32 columns
static_assert(kTmemA + 32 * kPA * kSA <= 512, "tensor memory");
constexpr int kChunk = 4;                  // k-stages per staged chunk of codes
constexpr int kStgCodes = 128 * 128;       // 128 rows x 128 bytes of codes (4 stages)
constexpr int kStgSB = 128 * kChunk * 8;   // per row and stage: scale word, bias word
constexpr int kStgBuf = kStgCodes + kStgSB;
constexpr int kNStg = 4;                   // staged chunks at most: one being read, the rest in flight
constexpr int kEpiBytes = 16384;           // down: 4 warps x 32 x 32 fp32; gate_up: h rows

// Shared-memory layout of one pf_gemm instantiation (offsets 1024-aligned
// where the 128B swizzle needs it).  Router: six stages of A (128 router
// rows) and B (128 token rows).  Expert GEMMs: three stages of B (up to
// kStageRows token rows: one or more k-panels of a tile) and the staged
// code chunks; A lives in TMEM.
template <int MODE>
struct Lay {
  static constexpr int nSB = MODE == MODE_ROUTER ? kSB : 3;
  static constexpr int stageB = MODE == MODE_ROUTER ? 128 * 128 : kStageRows * 128;
  static constexpr int offA = nSB * stageB;
  static constexpr int offStg = offA + (MODE == MODE_ROUTER ? nSB * 128 * 128 : 0);
  static constexpr int offEpi = offStg + (MODE == MODE_ROUTER ? 0 : kNStg * kStgBuf);
  static constexpr int offTile = offEpi + kEpiBytes;
  static constexpr int offBars = offTile + 2 * kPfTileN * 4;
  static constexpr int smem = offBars + 512 + 1024;  // + alignment slack
  static constexpr int accCols = MODE == MODE_ROUTER ? 256 : kAccCols;
  static_assert(smem <= 227 * 1024, "shared memory");
  static_assert(stageB % 1024 == 0 && offA % 1024 == 0, "swizzled stages");
};

struct WsBars {
  uint64_t full_b[kSB], empty_b[kSB], full_a[kSA], empty_a[kSA], acc_full[2], acc_empty[2], drain;
  uint32_t tmem;
};

template <int MODE>
__device__ __forceinline__ int ws_num_tiles(const PfParams &P) {
  if constexpr (MODE == MODE_ROUTER)
    return ((P.E + 127) / 128) * ((P.t + 127) / 128);
  else
    return P.nitems[MODE == MODE_GATE_UP ? 0 : 1];
}

template <int MODE>
__device__ __forceinline__ int ws_nk(const PfParams &P) {
  return MODE == MODE_ROUTER ? 2 * P.H / 64 : (MODE == MODE_GATE_UP ? P.H / 64 : P.I / 64);
}

// Work item of tile ti.  Callers load items a tile or two before they use
// them, so that no role waits on a descriptor load.
template <int MODE>
__device__ __forceinline__ PfItem ws_item(const PfParams &P, int ti) {
  if constexpr (MODE == MODE_ROUTER) {
    const int nmt = (P.E + 127) / 128;
    PfItem it;
    it.g = 0, it.mt = ti % nmt, it.n0 = (ti / nmt) * 128;
    it.nlen = min(128, P.t - it.n0);
    it.rec = 0;
    return it;
  } else {
    return (MODE == MODE_GATE_UP ? P.items1 : P.items2)[ti];
  }
}

__device__ __forceinline__ int tile_n(const PfItem &it) { return (it.nlen + 15) & ~15; }

// Token rows a B stage loads per k-panel for N columns: 128-row boxes, then
// 32-row boxes for the rest.
__device__ __forceinline__ int panel_rows(int N) { return (N & ~127) + (((N & 127) + 31) & ~31); }

// k-panels per B stage (expert GEMMs): a narrow tile carries several panels
// in one stage buffer, so that each TMA round trip (a latency of thousands
// of cycles) feeds more MMAs.  A divisor of nk.
__device__ __forceinline__ int panels_per_stage(int N, int nk) {
  const int r = panel_rows(N);
  for (int p = 4; p > 1; p >>= 1)
    if (p * r <= kStageRows && nk % p == 0) return p;
  return 1;
}

template <int MODE>
__device__ __forceinline__ bool item_ok(const PfItem &it) {
  return MODE == MODE_ROUTER || (it.rec != 0 && (it.rec & 15u) == 0);
}

// lane 0 waits, the warp learns the outcome
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t par, const PfParams &P) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = pf_wait(bar, par, P);
  return __shfl_sync(FULLM, ok ? 1 : 0, 0) != 0;
}

// Weight row of tile row r.  A gate_up tile covers 64 intermediate indices
// mt*64 .. mt*64+63: each 32-row quadrant q holds the gate rows of indices
// 16q .. 16q+15 followed by their up rows, so that the epilogue finds gate i
// and up i in lanes l and l + 16 of one warp.  A down tile: 128 output rows.
// (Row parity = parity of r in both layouts.)
template <int MODE>
__device__ __forceinline__ int ws_weight_row(const PfParams &P, int mt, int r) {
  if constexpr (MODE == MODE_GATE_UP)
    return ((r & 16) ? P.I : 0) + mt * 64 + 16 * (r >> 5) + (r & 15);
  else
    return mt * 128 + r;
}

// Global sources of one staging thread t for a tile, formed once per tile:
// its four 16-byte code segments (row (i * 256 + t) / 8, piece t % 8, at
// k-panel 0; a chunk's row segment is 32 * bits bytes, so pieces past
// 2 * bits are not copied) and the scale / bias entries of row t % 128.
// w16 (input width a multiple of 256): every row's scale and bias tables
// start on an 8-byte boundary, so a chunk's four entries of a table (8
// bytes) lie in one aligned 16-byte window; thread t then copies that
// window of table t / 128 (s: its row's table at k-panel 0).
struct StgRows {
  const uint8_t *c[4];
  const uint8_t *s, *b;
  int seg;  // bytes of a row per chunk of four k-panels
  bool ok, w16;
};

// code width of a tile's record: the shared expert's is 4-bit; LB: the
// routed records may be narrower (else every record is 4-bit)
template <bool LB>
__device__ __forceinline__ int item_bits(const PfParams &P, const PfItem &it) {
  return LB && it.g != P.E ? P.bits : 4;
}

template <int MODE, bool LB>
__device__ __forceinline__ StgRows stage_rows(const PfParams &P, const PfItem &it, int t) {
  StgRows sr{};
  sr.ok = item_ok<MODE>(it);
  if (sr.ok) {
    const uint8_t *rec = reinterpret_cast<const uint8_t *>(it.rec);
    const QOff q = it.g == P.E ? (MODE == MODE_GATE_UP ? P.sgu : P.sdn) : (MODE == MODE_GATE_UP ? P.gu : P.dn);
    const int inp = MODE == MODE_GATE_UP ? P.H : P.I;
    const int bits = item_bits<LB>(P, it);
    sr.seg = 32 * bits;
#pragma unroll
    for (int i = 0; i < 4; i++) {
      const int idx = i * 256 + t, row = idx >> 3, part = idx & 7;
      sr.c[i] = part < 2 * bits
                    ? rec + q.w + (size_t)ws_weight_row<MODE>(P, it.mt, row) * (inp / 8 * bits) + part * 16
                    : nullptr;
    }
    const size_t g2 = (size_t)ws_weight_row<MODE>(P, it.mt, t & 127) * (inp / 64) * 2;
    sr.w16 = (inp & 255) == 0;
    sr.s = rec + (sr.w16 && t >= 128 ? q.b : q.s) + g2;
    sr.b = rec + q.b + g2;
  }
  return sr;
}

// Stage one chunk of codes (k-panels 4kc .. 4kc+3 of a tile) into shared
// memory, by the 256 producer threads (t): 128 rows x 128 bytes, copied by 8
// threads per row segment so that each warp instruction reads four whole
// 128-byte lines (16-byte pieces placed at piece ^ (row & 7) against bank
// conflicts); plus the scale and bias entries: w16, per row and table the
// 16-byte window holding the chunk's four entries (scales at row * 16,
// biases 2048 bytes further); otherwise, per row and panel, the 4-byte words
// holding its scale and bias.  A segment or window may run past the end of
// a row, into bytes of the same record (codes are followed by the scale and
// bias tables, and a table's end is 16-byte aligned); those bytes are never
// used.
__device__ __forceinline__ void stage_chunk(const StgRows &sr, int kc, int nk, int t, uint8_t *buf) {
  if (sr.ok) {
#pragma unroll
    for (int i = 0; i < 4; i++) {
      const int idx = i * 256 + t, row = idx >> 3, part = idx & 7;
      if (sr.c[i]) tc05::cp16(buf + row * 128 + ((part ^ (row & 7)) << 4), sr.c[i] + kc * sr.seg);
    }
    const int r = t & 127;
    if (sr.w16) {
      tc05::cp16(buf + kStgCodes + (t >> 7) * 2048 + r * 16,
                 reinterpret_cast<const uint8_t *>(((uintptr_t)sr.s + 8 * kc) & ~(uintptr_t)15));
      tc05::cp_commit();
      return;
    }
#pragma unroll
    for (int v = 0; v < 2; v++) {
      const int u = 2 * (t >> 7) + v;
      const int kk = min(kc * kChunk + u, nk - 1);
      tc05::cp4(buf + kStgCodes + (r * kChunk + u) * 8,
                reinterpret_cast<const uint8_t *>((uintptr_t)(sr.s + kk * 2) & ~(uintptr_t)3));
      tc05::cp4(buf + kStgCodes + (r * kChunk + u) * 8 + 4,
                reinterpret_cast<const uint8_t *>((uintptr_t)(sr.b + kk * 2) & ~(uintptr_t)3));
    }
  }
  tc05::cp_commit();
}

// Scale and bias (bf16 bits, in .x and .y) of row r, k-panel u of a staged
// chunk.  w16: the chunk's entries sit at byte sel (0 or 8) of the row's
// 16-byte windows; otherwise in half sel of the panel's 4-byte words.
__device__ __forceinline__ uint2 staged_sb(const uint8_t *buf, int r, int u, uint32_t sel, bool w16) {
  if (w16) {
    const uint8_t *p = buf + kStgCodes + r * 16 + sel + 2 * u;
    return make_uint2(*reinterpret_cast<const uint16_t *>(p), *reinterpret_cast<const uint16_t *>(p + 2048));
  }
  const uint2 w = *reinterpret_cast<const uint2 *>(buf + kStgCodes + (r * kChunk + u) * 8);
  return make_uint2((w.x >> (16 * sel)) & 0xffffu, (w.y >> (16 * sel)) & 0xffffu);
}

// Row r's 64 codes of k-panel u of a staged chunk -> bf16(scale * code +
// bias), k permuted within 8-blocks, as 32 words of two bf16 each (the row's
// 32 A columns of the panel).  4-bit records; ws_dequant_row_lb below takes
// 2- and 3-bit ones into the same layout.  sb: the panel's scale and bias.
__device__ __forceinline__ void ws_dequant_row(const uint8_t *buf, int r, int u, uint2 sb, uint32_t (&a)[32]) {
  const uint32_t s2 = sb.x * 0x10001u, b2 = sb.y * 0x10001u;
#pragma unroll
  for (int hf = 0; hf < 2; hf++) {
    const uint4 c = *reinterpret_cast<const uint4 *>(buf + r * 128 + (((2 * u + hf) ^ (r & 7)) << 4));
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int ch = 0; ch < 4; ch++)
#pragma unroll
      for (int j = 0; j < 4; j++) {
        const uint32_t v = ((w[ch] >> (4 * j)) & 0x000f000fu) | 0x43004300u;  // (128 + n_j, 128 + n_{j+4})
        const uint32_t qv = bfma2(v, 0x3f803f80u, 0xc300c300u);              // the codes, exact
        a[16 * hf + 4 * ch + j] = bfma2(qv, s2, b2);                         // bf16(s*q + b)
      }
  }
}

// ws_dequant_row for B = 2 or 3: the panel's 8B code bytes sit at byte 8Bu of
// the row's staged segment (8-byte loads never straddle a 16-byte piece);
// word 4ch + j of the output pairs codes 8ch + j and 8ch + j + 4, as for 4
// bits.  Each half of the panel (32 codes, B words) goes through the decode
// codec's CodecO4<B>, which puts every such pair at shift 0 on 128.0 (a byte
// permute per 16 codes for 2 bits, a funnel shift and a bit select per 24-bit
// window for 3), so a pair costs one shift and one mask-or.
template <int B>
__device__ __forceinline__ void ws_dequant_row_lb(const uint8_t *buf, int r, int u, uint2 sb, uint32_t (&a)[32]) {
  const uint32_t s2 = sb.x * 0x10001u, b2 = sb.y * 0x10001u;
  uint32_t w[2 * B];
#pragma unroll
  for (int k = 0; k < B; k++) {
    const int byte = 8 * B * u + 8 * k;
    const uint2 q = *reinterpret_cast<const uint2 *>(buf + r * 128 + (((byte >> 4) ^ (r & 7)) << 4) + (byte & 15));
    w[2 * k] = q.x, w[2 * k + 1] = q.y;
  }
#pragma unroll
  for (int h = 0; h < 2; h++) {
    uint32_t hw[B], v[16];
#pragma unroll
    for (int k = 0; k < B; k++) hw[k] = w[B * h + k];
    CodecO4<B>::unpack(hw, v);  // v[4g + j] = (128 + code 8g + j, 128 + code 8g + j + 4) of the half
#pragma unroll
    for (int i = 0; i < 16; i++) {
      const uint32_t qv = bfma2(v[i], 0x3f803f80u, 0xc300c300u);  // the codes, exact
      a[16 * h + i] = bfma2(qv, s2, b2);                         // bf16(s*q + b)
    }
  }
}

__device__ __forceinline__ void dequant_row_bits(int bits, const uint8_t *buf, int r, int u, uint2 sb,
                                                 uint32_t (&a)[32]) {
  if (bits == 4)
    ws_dequant_row(buf, r, u, sb, a);
  else if (bits == 3)
    ws_dequant_row_lb<3>(buf, r, u, sb, a);
  else
    ws_dequant_row_lb<2>(buf, r, u, sb, a);
}

template <int MODE, bool LB = false>
__global__ void __launch_bounds__(kWsThreads, 1) pf_gemm(const __grid_constant__ PfParams P) {
  pdl_launch_next();
  extern __shared__ __align__(1024) uint8_t smraw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~(uintptr_t)1023);
  using LY = Lay<MODE>;
  WsBars &B = *reinterpret_cast<WsBars *>(sm + LY::offBars);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < LY::nSB; s++) {
      mbar_init(&B.full_b[s], 1);
      mbar_init(&B.empty_b[s], 1);
    }
    for (int s = 0; s < kSA; s++) {
      mbar_init(&B.full_a[s], 4);  // the four warps of one dequant group
      mbar_init(&B.empty_a[s], 1);
    }
    for (int b = 0; b < 2; b++) {
      mbar_init(&B.acc_full[b], 1);
      mbar_init(&B.acc_empty[b], 4);
    }
    mbar_init(&B.drain, 1);
    fence_mbar_init();
  }
  if (warp == 0) tc05::alloc(&B.tmem, 512);
  tc05::fence_before();
  __syncthreads();
  tc05::fence_after();
  const uint32_t tmem = B.tmem;
  // the setup above overlaps the previous kernel's end; everything below may
  // read earlier kernels' results (the work-list sizes among them)
  pdl_wait_prev();
  const int ntiles = ws_num_tiles<MODE>(P);
  const int nk = ws_nk<MODE>(P);
  const int my_tiles = (int)blockIdx.x < ntiles ? (ntiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  auto tile_of = [&](int lt) { return (int)blockIdx.x + lt * (int)gridDim.x; };

  if (warp == 0) {
    // ---------------------------------------------------------------- MMA issue
    // The whole warp walks the loop (warp-uniform state, waits by lane 0 with
    // the outcome broadcast); one elected lane issues each MMA group and
    // commit.  Ring positions and phases are kept incrementally: this loop is
    // on the critical path.
    {
      int sa = 0, sb = 0;
      uint32_t pa = 0, pb = 0;
      bool ok = true;
      PfItem nx{};
      const uint64_t desc0 = tc05::sdesc(smem_u32(sm));  // + (byte offset >> 4) within shared memory
      if (my_tiles > 0) nx = ws_item<MODE>(P, tile_of(0));
      for (int lt = 0; lt < my_tiles && ok; lt++) {
        const PfItem cur = nx;
        if (lt + 1 < my_tiles) nx = ws_item<MODE>(P, tile_of(lt + 1));
        const int b = lt & 1;
        if (!warp_wait(&B.acc_empty[b], (uint32_t)(((lt >> 1) & 1) ^ 1), P)) {
          ok = false;
          break;
        }
        tc05::fence_after();
        const uint32_t d = tmem + (uint32_t)(b * LY::accCols);
        const int N = tile_n(cur);
        const uint32_t idesc = tc05::idesc_bf16(N);
        const int ppb = MODE == MODE_ROUTER ? 1 : panels_per_stage(N, nk);
        const uint32_t pstep = (uint32_t)(panel_rows(N) * 128) >> 4;  // descriptor step per panel
        int pp = 0, ap = 0;  // panel within the B stage, within the A stage
        uint64_t bdesc = desc0;
        for (int kk = 0; kk < nk; kk++) {
          if (pp == 0) {
            if (!warp_wait(&B.full_b[sb], pb, P)) {
              ok = false;
              break;
            }
            bdesc = desc0 + (uint32_t)(sb * LY::stageB >> 4);
          }
          if constexpr (MODE == MODE_ROUTER) {
            tc05::fence_after();
            const uint64_t adesc = desc0 + (uint32_t)((LY::offA + sb * 128 * 128) >> 4);
            if (tc05::elect_one()) {
#pragma unroll
              for (int j = 0; j < 4; j++) tc05::mma(d, adesc + 2 * j, bdesc + 2 * j, idesc, (kk | j) != 0);
            }
            __syncwarp();
          } else {
            if (ap == 0 && !warp_wait(&B.full_a[sa], pa, P)) {
              ok = false;
              break;
            }
            tc05::fence_after();
            const bool last = ap == kPA - 1 || kk == nk - 1;  // the A stage's last panel
            if (tc05::elect_one()) {
              tc05::mma_ts_k64(d, tmem + (uint32_t)(kTmemA + 32 * (kPA * sa + ap)), bdesc, idesc, kk != 0);
              if (last) tc05::commit(&B.empty_a[sa]);
            }
            __syncwarp();
            if (last) {
              ap = 0;
              if (++sa == kSA) sa = 0, pa ^= 1;
            } else {
              ap++;
            }
          }
          bdesc += pstep;
          if (++pp == ppb) {
            if (tc05::elect_one()) tc05::commit(&B.empty_b[sb]);
            __syncwarp();
            pp = 0;
            if (++sb == LY::nSB) sb = 0, pb ^= 1;
          }
        }
        if (ok) {
          if (tc05::elect_one()) tc05::commit(&B.acc_full[b]);
          __syncwarp();
        }
      }
      // every MMA issued here has completed before TMEM is released
      if (tc05::elect_one()) tc05::commit(&B.drain);
      __syncwarp();
      warp_wait(&B.drain, 0, P);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- B producer (TMA)
    // router: 128 token rows of x^ hi / lo and the 128 router rows; gate_up
    // and down: the tile's rows of the grouped operand (x^ rows gathered in
    // group order, or h), boxes of 128 rows then 32-row boxes for the tail
    int f = 0;  // B stages
    PfItem ia{}, ib{};
    if (my_tiles > 0) ia = ws_item<MODE>(P, tile_of(0));
    bool ok = true;
    for (int lt = 0; lt < my_tiles && ok; lt++) {
      if (lt + 1 < my_tiles) ib = ws_item<MODE>(P, tile_of(lt + 1));
      const int N = tile_n(ia);
      const int n128 = N >> 7, n32 = ((N & 127) + 31) >> 5, nops = n128 + n32;
      const int ppb = MODE == MODE_ROUTER ? 1 : panels_per_stage(N, nk), prow = panel_rows(N);
      const uint32_t bytes = MODE == MODE_ROUTER ? (uint32_t)(2 * 128 * 128) : (uint32_t)(ppb * prow * 128);
      const CUtensorMap *m128 = MODE == MODE_GATE_UP ? &P.tm_xc : &P.tm_h;
      const CUtensorMap *m32 = MODE == MODE_GATE_UP ? &P.tm_xc32 : &P.tm_h32;
      const int ent = P.t * (P.K + 1);  // rows of one k-panel of xc / h
      for (int kk = 0; kk < nk; kk += ppb, f++) {
        const int s = f % LY::nSB;
        if (!warp_wait(&B.empty_b[s], (uint32_t)(((f / LY::nSB) & 1) ^ 1), P)) {
          ok = false;
          break;
        }
        uint8_t *sb = sm + s * LY::stageB;
        if (lane == 0) mbar_expect_tx(&B.full_b[s], bytes);
        __syncwarp();
        if constexpr (MODE == MODE_ROUTER) {
          const int nq = P.H / 64, kq = kk % nq, yb = (kk < nq ? 0 : P.t) + ia.n0;
          if (lane == 0) {
            tc05::tma_load_2d(sm + LY::offA + s * 128 * 128, &P.tm_router, kq * 64, ia.mt * 128, &B.full_b[s]);
            tc05::tma_load_2d(sb, &P.tm_xr, kq * 64, yb, &B.full_b[s]);
          }
        } else {
          // k-panels kk .. kk+ppb-1, one after another; in each the tile's
          // rows are contiguous (rows past the tile feed only accumulator
          // columns that are never stored).  Lane l: box l % nops of panel
          // l / nops.
          if (lane < ppb * nops) {
            const int pp = lane / nops, o = lane - pp * nops;
            const int r0 = o < n128 ? 128 * o : 128 * n128 + 32 * (o - n128);
            tc05::tma_load_2d(sb + (pp * prow + r0) * 128, o < n128 ? m128 : m32, 0, (kk + pp) * ent + ia.n0 + r0,
                              &B.full_b[s]);
          }
        }
      }
      ia = ib;
    }
    // copies still in flight land before the CTA ends: the last issue of
    // every stage (after a timeout the consumer may have stopped early, so
    // the earlier stages' copies need not have been waited for)
    if (lane == 0)
      for (int g = f > LY::nSB ? f - LY::nSB : 0; g < f; g++)
        pf_wait(&B.full_b[g % LY::nSB], (uint32_t)((g / LY::nSB) & 1), P);
    __syncwarp();
  } else if (warp < 10) {
    // ---------------------------------------------------------------- A producers
    if constexpr (MODE != MODE_ROUTER) {
      // thread t stages codes; thread (warp, lane) dequantizes tile row
      // r = 32 * (warp % 4) + lane (the TMEM lanes its warp may write); warp
      // group hf fills the chunk's A stage hf (k-panels 2hf, 2hf + 1)
      const int t = tid - 64, r = 32 * (warp & 3) + lane, hf = (warp - 2) >> 2;
      // staging depth: four chunks for 4-bit records; the funnel-shift
      // dequant of narrower ones ran slower with the fourth (measured)
      constexpr int NStg = LB ? 3 : kNStg;
      const int nct = (nk + kChunk - 1) / kChunk;  // chunks per tile
      const int total = my_tiles * nct;
      const int inp = MODE == MODE_GATE_UP ? P.H : P.I;
      uint8_t *stg = sm + LY::offStg;
      // items of the staging position's tile and of the tile after it
      PfItem snext{};
      StgRows srow{};
      int slt = 0;
      if (my_tiles > 0) srow = stage_rows<MODE, LB>(P, ws_item<MODE>(P, tile_of(0)), t);
      if (my_tiles > 1) snext = ws_item<MODE>(P, tile_of(1));
      auto issue = [&](int c) {
        if (c >= total) {
          tc05::cp_commit();  // empty group keeps the group count uniform
          return;
        }
        const int lt = c / nct;
        if (lt != slt) {
          srow = stage_rows<MODE, LB>(P, lt == slt + 1 ? snext : ws_item<MODE>(P, tile_of(lt)), t);
          slt = lt;
          if (lt + 1 < my_tiles) snext = ws_item<MODE>(P, tile_of(lt + 1));
        }
        stage_chunk(srow, c - lt * nct, nk, t, stg + (c % NStg) * kStgBuf);
      };
      for (int c = 0; c < NStg - 1; c++) issue(c);
      // parity of the weight row = parity of r (tile row bases are even):
      // rodd tells whether the row's tables start in the second half of a
      // 4-byte word, rodd8 (w16) in the second half of a 16-byte window
      const bool w16 = (inp & 255) == 0;
      const uint32_t rodd = (uint32_t)(r & (inp / 64) & 1), rodd8 = (uint32_t)(r & (inp / 256) & 1);
      int qlt = -1, qbits = 4;  // the tile being dequantized and its code width
      bool ok = true;
      for (int c = 0; c < total && ok; c++) {
        tc05::cp_wait_group<NStg - 2>();  // this thread's copies of chunk c are done
        tc05::named_sync(3, 256);  // everyone's are; everyone is done reading chunk c - 1
        // the second group, which waits longer for its A stage, issues chunk
        // c + NStg - 1 (into chunk c - 1's buffer) before that wait; the first
        // group after its dequantization
        if (hf) issue(c + NStg - 1);
        const int lt = c / nct, kc = c - lt * nct;
        const uint8_t *buf = stg + (c % NStg) * kStgBuf;
        const int ns = min(kChunk, nk - kc * kChunk);
        if (LB && lt != qlt) qbits = item_bits<LB>(P, ws_item<MODE>(P, tile_of(lt))), qlt = lt;
        const int u0 = kPA * hf;  // this group's A stage of the chunk, if the chunk has it
        if (u0 < ns) {
          // A stage ga of this CTA's sequence ((nk + kPA - 1) / kPA stages a tile)
          const int ga = lt * ((nk + kPA - 1) / kPA) + (kc * kChunk + u0) / kPA, sa = ga % kSA;
          if (warp_wait(&B.empty_a[sa], (uint32_t)(((ga / kSA) & 1) ^ 1), P)) {
            tc05::fence_after();  // after the MMAs that read this A stage
            const uint32_t ta = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(kTmemA + 32 * kPA * sa);
            // scale / bias of entry row * G + kk: its place in the staged windows or words
            const int kk0 = kc * kChunk + u0;
            uint32_t av0[32], av1[32];
            const uint32_t sel8 = 8u * ((rodd8 + (uint32_t)kc) & 1u);
            const uint2 sb0 = staged_sb(buf, r, u0, w16 ? sel8 : (rodd + (uint32_t)kk0) & 1u, w16);
            if (LB) dequant_row_bits(qbits, buf, r, u0, sb0, av0);
            else ws_dequant_row(buf, r, u0, sb0, av0);
            tc05::st32(ta, av0);
            if (u0 + 1 < ns) {
              const uint2 sb1 = staged_sb(buf, r, u0 + 1, w16 ? sel8 : (rodd + (uint32_t)kk0 + 1u) & 1u, w16);
              if (LB) dequant_row_bits(qbits, buf, r, u0 + 1, sb1, av1);
              else ws_dequant_row(buf, r, u0 + 1, sb1, av1);
              tc05::st32(ta + 32, av1);
            }
            tc05::wait_st();
            tc05::fence_before();
            __syncwarp();
            // (failure-detection test: one warp of CTA 0 withholds its
            // arrive on the first A stage of the gate_up GEMM, so that the
            // MMA warp's bounded wait runs out and every wait after it too)
            const bool withheld = MODE == MODE_GATE_UP && P.withhold && blockIdx.x == 0 && c == 0 && warp == 2;
            if (lane == 0 && !withheld) tc05::mbar_arrive(&B.full_a[sa]);
          } else {
            ok = false;
          }
        }
        // chunk c + NStg - 1 into chunk c - 1's buffer (free since the barrier
        // above), after this chunk's dequantization: its copies land chunks
        // before they are read, and their issue waits on the load queue
        if (!hf) issue(c + NStg - 1);
        // the eight producer warps stop together (they share a named barrier)
        ok = tc05::named_and(4, 256, ok);
      }
      tc05::cp_wait_group<0>();  // nothing in flight into shared memory at the end
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;    // TMEM lane quadrant this warp may read
    const int et = tid - 320;  // 0..127 over the epilogue warps
    int *trow = reinterpret_cast<int *>(sm + LY::offTile);
    float *twt = reinterpret_cast<float *>(sm + LY::offTile) + kPfTileN;
    PfItem nx{};
    unsigned hcnt = 0;  // gate_up: h chunks written so far (their buffers alternate)
    int pr[2] = {0, 0};
    float pw[2] = {0.f, 0.f};
    auto fetch_entries = [&](const PfItem &it) {  // down: this thread's two entries of a tile
#pragma unroll
      for (int h = 0; h < 2; h++) {
        const int j = et + 128 * h;  // entries past kPfTileN do not exist
        pr[h] = j < it.nlen ? P.rows[it.n0 + j] : 0;
        pw[h] = j < it.nlen ? P.wts[it.n0 + j] : 0.f;
      }
    };
    if (my_tiles > 0) {
      nx = ws_item<MODE>(P, tile_of(0));
      if (MODE == MODE_DOWN) fetch_entries(nx);
    }
    for (int lt = 0; lt < my_tiles; lt++) {
      const PfItem T = nx;
      if (lt + 1 < my_tiles) nx = ws_item<MODE>(P, tile_of(lt + 1));
      const int N = tile_n(T);
      const int b = lt & 1;
      if (MODE == MODE_DOWN) {
        tc05::named_sync(1, 128);  // the previous tile's readers are done
#pragma unroll
        for (int h = 0; h < 2; h++)
          if (et + 128 * h < kPfTileN) trow[et + 128 * h] = pr[h], twt[et + 128 * h] = pw[h];
        tc05::named_sync(1, 128);
      }
      // the four epilogue warps stop together (they share named barriers)
      if (!tc05::named_and(2, 128, warp_wait(&B.acc_full[b], (uint32_t)((lt >> 1) & 1), P))) break;
      tc05::fence_after();
      const uint32_t tl = tmem + (uint32_t)(b * LY::accCols) + ((uint32_t)(32 * q) << 16);
      if (item_ok<MODE>(T)) {
        for (int c0 = 0; c0 < N; c0 += 32) {
          float v[32];
          tc05::ld32(tl + c0, v);
          if constexpr (MODE == MODE_ROUTER) {
            const int e = T.mt * 128 + 32 * q + lane;
            if (e < P.E)
#pragma unroll
              for (int j = 0; j < 32; j++)
                if (c0 + j < T.nlen) P.logits[(size_t)(T.n0 + c0 + j) * P.E + e] = v[j];
          } else if constexpr (MODE == MODE_DOWN) {
            // transpose the warp's 32 rows x 32 tokens through shared memory,
            // then one 16-byte reduction per (token, 4 rows)
            float *tb = reinterpret_cast<float *>(sm + LY::offEpi) + (warp - 10) * 1024;
#pragma unroll
            for (int j = 0; j < 32; j++) tb[j * 32 + lane] = v[j];
            __syncwarp();
            const int a = lane & 7, jj = lane >> 3;
            const int o = T.mt * 128 + 32 * q + 4 * a;
#pragma unroll
            for (int p = 0; p < 8; p++) {
              const int j = 4 * p + jj, col = c0 + j;
              if (col < T.nlen) {
                const float4 y = *reinterpret_cast<const float4 *>(tb + j * 32 + 4 * a);
                const float w = twt[col];
                tc05::red_add_v4(P.Y + (size_t)trow[col] * P.H + o, w * y.x, w * y.y, w * y.z, w * y.w);
              }
            }
            __syncwarp();
          } else {
            // lanes l < 16 hold gate, lanes l + 16 up, of index i = 16q + (l & 15):
            // the gate lane takes columns 0..15, the up lane 16..31, each
            // fetching the partner's value with one exchange per column
            const int up = lane >> 4, i = 16 * q + (lane & 15);
            uint16_t *hs = reinterpret_cast<uint16_t *>(sm + LY::offEpi) + (hcnt++ & 1) * (32 * 64);
#pragma unroll
            for (int j = 0; j < 16; j++) {
              const float mine = up ? v[16 + j] : v[j];
              const float other = __shfl_xor_sync(FULLM, up ? v[j] : v[16 + j], 16);
              const float g = up ? other : mine, u = up ? mine : other;
              const float h = __fdividef(g, 1.f + __expf(-g)) * u;
              hs[(16 * up + j) * 64 + (i & ~7) + perm8(i & 7)] = (uint16_t)f2bf_rn(h);
            }
            tc05::named_sync(1, 128);  // h of 32 tokens x 64 indices complete (buffers alternate)
            for (int k = et; k < 32 * 8; k += 128) {
              const int j = k >> 3, c = k & 7;
              if (c0 + j < T.nlen)
                *reinterpret_cast<uint4 *>(P.hbuf + ((size_t)T.mt * P.t * (P.K + 1) + T.n0 + c0 + j) * 64 + c * 8) =
                    *reinterpret_cast<const uint4 *>(hs + j * 64 + c * 8);
            }
          }
        }
      } else if (et == 0) {
        atomicCAS(P.status, 0, kStatusDevice);
      }
      if (MODE == MODE_DOWN && lt + 1 < my_tiles) fetch_entries(nx);
      tc05::fence_before();
      __syncwarp();
      if (lane == 0) tc05::mbar_arrive(&B.acc_empty[b]);
    }
  }

  tc05::fence_before();
  __syncthreads();
  if (warp == 0) tc05::dealloc(tmem, 512);
}

// Expert operand rows in group order, in k-panels: panel p holds elements
// 64p .. 64p+63 of the x^ row of every grouped entry e (warp per entry,
// 16-byte copies).  One k-stage of a gate_up tile's B is then one contiguous
// block of its rows x 128 bytes.  (h uses the same layout for the down GEMM.)
__global__ void pf_gather(const __grid_constant__ PfParams P) {
  pdl_begin();
  const int e = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  const int G = P.E + (P.sgate ? 1 : 0);
  if (e >= P.offs[G]) return;
  const uint4 *src = reinterpret_cast<const uint4 *>(P.xg + (size_t)P.rows[e] * P.H);
  const size_t ent = (size_t)P.t * (P.K + 1);
  // piece i (8 elements) of the row goes to k-panel i / 8; a lane's loads
  // of up to eight pieces are all in flight before its stores
  for (int i0 = 0; i0 < P.H / 8; i0 += 8 * 32) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; u++) {
      const int i = i0 + u * 32 + lane;
      if (i < P.H / 8) v[u] = src[i];
    }
#pragma unroll
    for (int u = 0; u < 8; u++) {
      const int i = i0 + u * 32 + lane;
      if (i < P.H / 8) reinterpret_cast<uint4 *>(P.xc + ((size_t)(i >> 3) * ent + e) * 64)[i & 7] = v[u];
    }
  }
}

// ------------------------------------------------------------ routing

// Unsigned key in the order of f; -0 is keyed as +0, so that a logit of -0
// ties with +0 (to the lower id) as the comparison of the two floats does
// (the tensor-core sum of an all-zero row's products may come out as -0).
__device__ __forceinline__ uint32_t orderable_f(float f) {
  const uint32_t u = __float_as_uint(f == 0.f ? 0.f : f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
// its inverse: the float a key was made from (bit for bit, but for -0)
__device__ __forceinline__ float from_orderable(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// One block per chunk of kPfChunk tokens, 16 warps of two tokens each:
// top-k (ties to the lower id) of E <= 1024 logits and softmax over the k
// chosen, per token; then the chunk's per-expert counts, gathered in a
// shared-memory histogram and stored once per expert (chist[e][chunk]), so
// that a popular expert's counter is not a global atomic every token hits.
// Lane l holds experts l, l + 32, ... (coalesced loads); each round takes
// the largest key, and among equal keys the lowest expert id.
// PM: keys per lane (E <= 32 PM).
constexpr int kTopkThreads = 512;
template <int PM>
__global__ void __launch_bounds__(kTopkThreads) pf_topk(const __grid_constant__ PfParams P) {
  pdl_begin();
  extern __shared__ int hist[];  // [E]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, c = blockIdx.x;
  const int E = P.E, K = P.K, nch = (P.t + kPfChunk - 1) / kPfChunk;
  for (int e = threadIdx.x; e < E; e += kTopkThreads) hist[e] = 0;
  __syncthreads();
  for (int j = 0; j < kPfChunk * 32 / kTopkThreads; j++) {
    const int tok = c * kPfChunk + j * (kTopkThreads / 32) + warp;
    if (tok >= P.t) break;  // warp-uniform
    const float *lg = P.logits + (size_t)tok * E;
    uint32_t key[PM];
#pragma unroll
    for (int i = 0; i < PM; i++) {
      const int e = i * 32 + lane;
      key[i] = e < E ? orderable_f(lg[e]) : 0u;
    }
    uint32_t bk = 0;
    int bi = 0;
#pragma unroll
    for (int i = 0; i < PM; i++)
      if (key[i] > bk) bk = key[i], bi = i;
    float myl = 0.f;
    int myid = 0;
    for (int r = 0; r < K; r++) {
      const uint32_t m = __reduce_max_sync(FULLM, bk);
      const uint32_t id = __reduce_min_sync(FULLM, bk == m ? (uint32_t)(bi * 32 + lane) : 0xffffffffu);
      if (lane == r) myid = (int)id, myl = from_orderable(m);  // the logit, from its key (no load)
      if (lane == (int)(id & 31)) {
        uint32_t nbk = 0;
        int nbi = 0;
#pragma unroll
        for (int i = 0; i < PM; i++) {
          if (i == bi) key[i] = 0u;
          if (key[i] > nbk) nbk = key[i], nbi = i;
        }
        bk = nbk, bi = nbi;
      }
    }
    const float mx = __shfl_sync(FULLM, myl, 0);
    const float ev = lane < K ? expf(myl - mx) : 0.f;
    const float z = warp_sum_f(ev);
    if (lane < K) {
      const float w = ev / z;
      P.tk_idx[(size_t)tok * K + lane] = myid;
      P.tk_w[(size_t)tok * K + lane] = w;
      if (P.topk_out) P.topk_out[(size_t)tok * K + lane] = (uint32_t)myid;
      if (P.topkw_out) P.topkw_out[(size_t)tok * K + lane] = w;
      atomicAdd(&hist[myid], 1);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kTopkThreads) P.chist[(size_t)e * nch + c] = hist[e];
}

// Block-wide exclusive scan (blockDim.x == 1024) of one int per thread.
__device__ int block_exscan(int v, int *sh, int *total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(FULLM, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh[w] = x;
  __syncthreads();
  if (w == 0) {
    int s = sh[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(FULLM, s, o);
      if (lane >= o) s += y;
    }
    sh[lane] = s;  // inclusive over warps
  }
  __syncthreads();
  const int r = x - v + (w ? sh[w - 1] : 0);
  *total = sh[31];
  __syncthreads();
  return r;
}

// Warp per expert e: its count (sum over token chunks) into counts[e], and
// in place the exclusive prefix of its chunk counts -- the place, within
// the expert's list, of each chunk's first entry.
__global__ void pf_group_count(const __grid_constant__ PfParams P) {
  pdl_begin();
  const int e = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (e >= P.E) return;
  const int nch = (P.t + kPfChunk - 1) / kPfChunk;
  int *h = P.chist + (size_t)e * nch;
  int base = 0;
  for (int k0 = 0; k0 < nch; k0 += 32) {
    const int k = k0 + lane;
    const int c = k < nch ? h[k] : 0;
    int x = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(FULLM, x, o);
      if (lane >= o) x += y;
    }
    if (k < nch) h[k] = base + x - c;
    base += __shfl_sync(FULLM, x, 31);
  }
  if (lane == 0) P.counts[e] = base;
}

// One block of 1024 threads.  Groups: the experts, then the shared expert
// with every token.  Exclusive scans of the group sizes and of their
// kPfTileN-token chunk counts give the group offsets and the chunk offsets
// (the tile work lists are written from them by pf_fill's blocks).
__global__ void __launch_bounds__(1024) pf_group(const __grid_constant__ PfParams P) {
  pdl_begin();
  __shared__ int s_off[1027], s_ch[1027], sh[32];
  const int E = P.E, G = E + (P.sgate ? 1 : 0);
  const int nmt1 = P.I / 64, nmt2 = P.H / 128;
  int m2[2], c2[2];
#pragma unroll
  for (int u = 0; u < 2; u++) {
    const int g = 2 * threadIdx.x + u;
    m2[u] = g < E ? P.counts[g] : (g < G ? P.t : 0);
    c2[u] = (m2[u] + kPfTileN - 1) / kPfTileN;
  }
  int tot_m, tot_ch;
  const int om = block_exscan(m2[0] + m2[1], sh, &tot_m);
  const int oc = block_exscan(c2[0] + c2[1], sh, &tot_ch);  // ends with a block barrier
#pragma unroll
  for (int u = 0; u < 2; u++) {
    const int g = 2 * threadIdx.x + u;
    if (g < G) {
      s_off[g] = u ? om + m2[0] : om;
      s_ch[g] = u ? oc + c2[0] : oc;
    }
  }
  if (threadIdx.x == 0) {
    s_off[G] = tot_m, s_ch[G] = tot_ch;
    P.nitems[0] = tot_ch * nmt1, P.nitems[1] = tot_ch * nmt2;
  }
  __syncthreads();
  for (int g = threadIdx.x; g <= G; g += blockDim.x) P.offs[g] = s_off[g];
  for (int g = threadIdx.x; g <= G; g += blockDim.x) P.choff[g] = s_ch[g];
}

// One block per chunk of kPfChunk tokens; its first warp gives the chunk's
// (token, expert) pairs, in token order, consecutive places in their
// experts' lists, so every list is in ascending token order (shared group:
// every token, weight = gate).  Then block c writes its share of the two
// GEMMs' tile work lists (item
// cc * nmt + mt: chunk cc of its group, row tile mt), each chunk's group
// found by a binary search over the chunk offsets.
constexpr int kFillThreads = 128;
__global__ void __launch_bounds__(kFillThreads) pf_fill(const __grid_constant__ PfParams P) {
  pdl_begin();
  extern __shared__ uint64_t fsm[];  // [G + 1] group records, then int [E] cnt, [G + 1] chunk and row offsets
  const int G = P.E + (P.sgate ? 1 : 0);
  uint64_t *srec = fsm;
  int *cnt = reinterpret_cast<int *>(srec + G + 1);  // [E] next place of each expert for this chunk
  int *sch = cnt + P.E, *soff = sch + G + 1;
  const int E = P.E, K = P.K, c = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
  // the work-list tables, by every thread (read after the barrier below)
  for (int g = tid; g <= G; g += kFillThreads) {
    srec[g] = g < E ? P.eaddr[g] : (g == E ? reinterpret_cast<uint64_t>(P.srec) : 0ull);
    sch[g] = P.choff[g];
    soff[g] = P.offs[g];
  }
  if (tid < 32) {
    // warp 0: the chunk's row lists
    const int nch = (P.t + kPfChunk - 1) / kPfChunk;
    for (int e = lane; e < E; e += 32) cnt[e] = P.offs[e] + P.chist[(size_t)e * nch + c];
    __syncwarp();
    const int t0 = c * kPfChunk, t1 = min(P.t, t0 + kPfChunk);
    // the chunk's (token, expert) pairs, eight rounds of 32 loaded at once
    for (int b0 = t0 * K; b0 < t1 * K; b0 += 8 * 32) {
      int ev[8];
      float wv[8];
#pragma unroll
      for (int j = 0; j < 8; j++) {
        const int i = b0 + j * 32 + lane;
        const bool v = i < t1 * K;
        ev[j] = v ? P.tk_idx[i] : -1;
        wv[j] = v ? P.tk_w[i] : 0.f;
      }
#pragma unroll
      for (int j = 0; j < 8; j++) {
        if (b0 + j * 32 >= t1 * K) break;  // warp-uniform
        const int i = b0 + j * 32 + lane;
        const bool v = i < t1 * K;
        const int e = ev[j];
        const unsigned peers = __match_any_sync(FULLM, e);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        const int base = v ? cnt[e] : 0;
        __syncwarp();
        if (v) {
          P.rows[base + rank] = i / K;
          P.wts[base + rank] = wv[j];
          if (rank == 0) cnt[e] = base + __popc(peers);
        }
        __syncwarp();
      }
    }
    if (P.sgate) {
      const int o = P.offs[E];
      for (int tok = t0 + lane; tok < t1; tok += 32) {
        P.rows[o + tok] = tok;
        P.wts[o + tok] = P.gam[tok];
      }
    }
  }
  __syncthreads();
  // every thread: this block's share of the two work lists
  const int nmt1 = P.I / 64, nmt2 = P.H / 128, n1 = P.nitems[0], total = n1 + P.nitems[1];
  const int per = (total + (int)gridDim.x - 1) / (int)gridDim.x, j1 = min(total, (c + 1) * per);
  for (int j = c * per + tid; j < j1; j += kFillThreads) {
    const bool first = j < n1;
    const int i = first ? j : j - n1, nmt = first ? nmt1 : nmt2;
    const int cc = i / nmt, mt = i - cc * nmt;
    int lo = 0, hi = G;  // the last group g with sch[g] <= cc holds chunk cc
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (sch[mid] <= cc) lo = mid; else hi = mid;
    }
    const int g = lo, ch = cc - sch[g], m = soff[g + 1] - soff[g];
    (first ? P.items1 : P.items2)[i] =
        PfItem{g, mt, soff[g] + ch * kPfTileN, min(kPfTileN, m - ch * kPfTileN), srec[g]};
  }
}

// out = bf16(Y (+ x)): four elements a thread per step when out is 8-byte
// aligned (x and Y always are; H is a multiple of 128), else one.
__global__ void pf_final(const __grid_constant__ PfParams P) {
  pdl_begin();
  const size_t n = (size_t)P.t * P.H, stride = (size_t)gridDim.x * blockDim.x;
  const size_t i0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const bool res = (P.flags & kResidualF) != 0;
  if ((reinterpret_cast<uintptr_t>(P.out) & 7u) == 0) {
    const float4 *y4 = reinterpret_cast<const float4 *>(P.Y), *x4 = reinterpret_cast<const float4 *>(P.x);
    uint2 *o2 = reinterpret_cast<uint2 *>(P.out);
    for (size_t i = i0; i < n / 4; i += stride) {
      float4 y = y4[i];
      if (res) {
        const float4 r = x4[i];
        y.x += r.x, y.y += r.y, y.z += r.z, y.w += r.w;
      }
      o2[i] = make_uint2(f2bf_rn(y.x) | f2bf_rn(y.y) << 16, f2bf_rn(y.z) | f2bf_rn(y.w) << 16);
    }
  } else {
    for (size_t i = i0; i < n; i += stride) {
      float y = P.Y[i];
      if (res) y += P.x[i];
      P.out[i] = (uint16_t)f2bf_rn(y);
    }
  }
}

size_t al(size_t n) { return (n + 1023) & ~(size_t)1023; }

// upper bound of the work items of one GEMM: sum over groups of
// ceil(m_g / kPfTileN) <= entries / kPfTileN + groups
size_t max_items(int E, int K, int t) {
  const size_t ent = (size_t)t * (K + 1);
  return ent / kPfTileN + (size_t)E + 2;
}

template <class F>
void carve(int H, int E, int K, int I, int t, F &&take) {
  const size_t ent = (size_t)t * (K + 1), nch = (size_t)((t + kPfChunk - 1) / kPfChunk);
  const size_t items = max_items(E, K, t);
  take(0, (size_t)2 * t * H * 2);  // xr_hi then xr_lo, adjacent
  take(1, 0);
  take(2, (size_t)t * H * 2);    // xg
  take(3, (size_t)t * 4);        // gam
  take(4, (size_t)t * E * 4);    // logits
  take(5, (size_t)t * K * 4);    // tk_idx
  take(6, (size_t)t * K * 4);    // tk_w
  take(7, nch * E * 4);          // chist
  take(8, (size_t)(E + 2) * 4);  // offs
  take(17, (size_t)(E + 2) * 4); // counts
  take(9, ent * 4);              // rows
  take(10, ent * 4);             // wts
  take(11, items * (I / 64) * sizeof(PfItem));
  take(12, items * (H / 128) * sizeof(PfItem));
  take(13, 64);                  // nitems
  take(14, ent * I * 2);         // hbuf
  take(15, (size_t)t * H * 4);   // Y
  take(16, ent * H * 2);         // xc
  take(18, (size_t)(E + 3) * 4); // choff
}

}  // namespace

size_t pf_workspace_bytes(int H, int E, int K, int I, int t) {
  size_t b = 0;
  carve(H, E, K, I, t, [&](int, size_t n) { b += al(n); });
  return b;
}

void pf_carve(PfParams &p, void *work) {
  char *base = reinterpret_cast<char *>(work);
  size_t o = 0;
  void *ptr[19];
  carve(p.H, p.E, p.K, p.I, p.t, [&](int k, size_t n) {
    ptr[k] = base + o;
    o += al(n);
  });
  p.xr_hi = (uint16_t *)ptr[0];
  p.xr_lo = p.xr_hi + (size_t)p.t * p.H;
  p.xg = (uint16_t *)ptr[2];
  p.gam = (float *)ptr[3];
  p.logits = (float *)ptr[4];
  p.tk_idx = (int *)ptr[5];
  p.tk_w = (float *)ptr[6];
  p.chist = (int *)ptr[7];
  p.offs = (int *)ptr[8];
  p.rows = (int *)ptr[9];
  p.wts = (float *)ptr[10];
  p.items1 = (PfItem *)ptr[11];
  p.items2 = (PfItem *)ptr[12];
  p.nitems = (int *)ptr[13];
  p.hbuf = (uint16_t *)ptr[14];
  p.Y = (float *)ptr[15];
  p.xc = (uint16_t *)ptr[16];
  p.counts = (int *)ptr[17];
  p.choff = (int *)ptr[18];
}

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return (EncodeTiledFn) nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// bf16 [rows][cols] row-major, box (64 columns = 128 bytes) x box_rows, 128B swizzle
// (a k-panel buffer is [cols / 64 * entries][64])
bool make_map(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int pf_tensor_maps(PfParams &p, const char **why) {
  const uint64_t H = (uint64_t)p.H, t = (uint64_t)p.t;
  if (!encode_fn()) {
    *why = "cuTensorMapEncodeTiled is not available from the driver";
    return -1;
  }
  const uint64_t ent = t * (uint64_t)(p.K + 1);
  if (!make_map(&p.tm_router, p.router, H, (uint64_t)p.E, 128) || !make_map(&p.tm_xr, p.xr_hi, H, 2 * t, 128) ||
      !make_map(&p.tm_h, p.hbuf, 64, (uint64_t)p.I / 64 * ent, 128) ||
      !make_map(&p.tm_h32, p.hbuf, 64, (uint64_t)p.I / 64 * ent, 32) ||
      !make_map(&p.tm_xc, p.xc, 64, H / 64 * ent, 128) || !make_map(&p.tm_xc32, p.xc, 64, H / 64 * ent, 32)) {
    *why = "cuTensorMapEncodeTiled rejected a tensor map";
    return -1;
  }
  return 0;
}

// A kernel of the chain after the first.  pdl: it may launch while the
// previous one ends (programmatic dependent launch; the kernel waits for it
// with griddepcontrol.wait before reading its results).  Only between two
// kernels: with an event recorded between them (the timed call) the launch
// keeps plain stream order, and griddepcontrol.wait has nothing to wait for.
template <class K>
cudaError_t launch_after(K kernel, int grid, int block, size_t smem, cudaStream_t st, bool pdl, const PfParams &p) {
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

cudaError_t pf_launch(PfParams &p, cudaStream_t st, cudaEvent_t const *events) {
  const int t = p.t, nch = (t + kPfChunk - 1) / kPfChunk;
  const size_t ent_cap = (size_t)t * (p.K + 1);
  cudaError_t e;
  auto mark = [&](int i) { return events ? cudaEventRecord(events[i], st) : cudaSuccess; };
  const bool pdl = events == nullptr;
  if ((e = cudaMemsetAsync(p.status, 0, 4, st))) return e;
  if (!p.route_only && (e = cudaMemsetAsync(p.Y, 0, (size_t)t * p.H * 4, st))) return e;
  if ((e = cudaFuncSetAttribute(pf_gemm<MODE_ROUTER>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Lay<MODE_ROUTER>::smem)))
    return e;
  if ((e = cudaFuncSetAttribute(pf_gemm<MODE_GATE_UP, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Lay<MODE_GATE_UP>::smem)))
    return e;
  if ((e = cudaFuncSetAttribute(pf_gemm<MODE_DOWN, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Lay<MODE_DOWN>::smem)))
    return e;
  if ((e = cudaFuncSetAttribute(pf_gemm<MODE_GATE_UP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Lay<MODE_GATE_UP>::smem)))
    return e;
  if ((e = cudaFuncSetAttribute(pf_gemm<MODE_DOWN>, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay<MODE_DOWN>::smem)))
    return e;
  const int ntr = ((p.E + 127) / 128) * ((t + 127) / 128);
  const int g_router = ntr < p.n_sms ? ntr : p.n_sms;
  if ((e = mark(0))) return e;
  pf_prep<<<t, 256, 0, st>>>(p);
  if ((e = mark(1))) return e;
  if ((e = launch_after(pf_gemm<MODE_ROUTER>, g_router, kWsThreads, Lay<MODE_ROUTER>::smem, st, pdl, p))) return e;
  if ((e = mark(2))) return e;
  const size_t hs = (size_t)p.E * 4;
  if (p.E <= 128)
    e = launch_after(pf_topk<4>, nch, kTopkThreads, hs, st, pdl, p);
  else if (p.E <= 256)
    e = launch_after(pf_topk<8>, nch, kTopkThreads, hs, st, pdl, p);
  else if (p.E <= 512)
    e = launch_after(pf_topk<16>, nch, kTopkThreads, hs, st, pdl, p);
  else
    e = launch_after(pf_topk<32>, nch, kTopkThreads, hs, st, pdl, p);
  if (e || (e = mark(3))) return e;
  if ((e = launch_after(pf_group_count, (p.E + 7) / 8, 256, 0, st, pdl, p)) || (e = mark(4))) return e;
  if ((e = launch_after(pf_group, 1, 1024, 0, st, pdl, p)) || (e = mark(5))) return e;
  if ((e = launch_after(pf_fill, nch, kFillThreads, (size_t)(p.E + 2) * 8 + (size_t)(3 * p.E + 6) * 4, st, pdl, p)) ||
      (e = mark(6)))
    return e;
  if (!p.route_only) {
    if ((e = launch_after(pf_gather, (int)((ent_cap + 7) / 8), 256, 0, st, pdl, p)) || (e = mark(7))) return e;
    e = p.bits == 4 ? launch_after(pf_gemm<MODE_GATE_UP>, p.n_sms, kWsThreads, Lay<MODE_GATE_UP>::smem, st, pdl, p)
                    : launch_after(pf_gemm<MODE_GATE_UP, true>, p.n_sms, kWsThreads, Lay<MODE_GATE_UP>::smem, st, pdl, p);
    if (e || (e = mark(8))) return e;
    e = p.bits == 4 ? launch_after(pf_gemm<MODE_DOWN>, p.n_sms, kWsThreads, Lay<MODE_DOWN>::smem, st, pdl, p)
                    : launch_after(pf_gemm<MODE_DOWN, true>, p.n_sms, kWsThreads, Lay<MODE_DOWN>::smem, st, pdl, p);
    if (e || (e = mark(9))) return e;
    if ((e = launch_after(pf_final, 1024, 256, 0, st, pdl, p)) || (e = mark(10))) return e;
  }
  return cudaGetLastError();
}

}  // namespace moe
