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
//           with all t tokens); per-chunk bases; tile work lists
//   fill    token lists in ascending token order (stable), routing weights
//   gate_up per (group, 64 gate + 64 up rows, <= 256 tokens): weights
//           dequantized to bf16 into 128B-swizzled shared memory (A), token
//           rows gathered (B), tcgen05 MMA into TMEM; epilogue
//           h = silu(gate) * up -> bf16
//   down    per (group, 128 output rows, <= 256 tokens): A = dequantized
//           down rows, B = h; epilogue Y[token] += weight * y (fp32)
//   final   out = bf16(Y) (+ x for a residual layer)
// The k order inside every 8-element block is permuted the same way on both
// expert operands so that one mask / FMA pair turns two codes into a bf16
// pair (nibbles j and j+4 of a code word share a register).
#include <cuda_runtime.h>

#include "prefill.cuh"
#include "tc05.cuh"

namespace moe {
namespace {

constexpr unsigned FULLM = 0xffffffffu;
constexpr uint32_t kResidualF = 1, kPrenormF = 2;
enum { MODE_ROUTER = 0, MODE_GATE_UP = 1, MODE_DOWN = 2 };

constexpr int kStageA = 128 * 128;       // 128 rows x 64 k bf16
constexpr int kStageB = kPfTileN * 128;  // 256 rows x 64 k bf16

__device__ __forceinline__ uint32_t f2bf_rn(float f) {
  uint32_t u = __float_as_uint(f);
  u += 0x7fffu + ((u >> 16) & 1u);
  return u >> 16;
}

// position of natural index j inside its 8-block under the operand
// permutation: pairs (0,4),(1,5),(2,6),(3,7) are adjacent
__device__ __forceinline__ int perm8(int j) { return (j & 3) * 2 + (j >> 2); }

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(FULLM, v, o);
  return v;
}

// bounded wait on an mbarrier phase; false (status set) once the limit passes
__device__ bool pf_wait(uint64_t *bar, uint32_t par, const PfParams &P) {
  if (mbar_try_wait(bar, par)) return true;
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, par)) {
    if (globaltimer() - t0 > P.timeout_ns) {
      atomicCAS(P.status, 0, kStatusTimeout);
      return false;
    }
  }
  return true;
}

// ------------------------------------------------------------ prep
// Block per token: x^, router operands (hi/lo, natural order), expert operand
// (bf16 of x^, permuted), shared gate sigmoid(sg . x^).
__global__ void pf_prep(const __grid_constant__ PfParams P) {
  __shared__ float red[32];
  const int tok = blockIdx.x, H = P.H, nw = blockDim.x >> 5;
  const float *xr = P.x + (size_t)tok * H;
  float scale = 1.f;
  if (P.flags & kPrenormF) {
    float ss = 0.f;
    for (int i = threadIdx.x; i < H; i += blockDim.x) ss += xr[i] * xr[i];
    ss = warp_sum_f(ss);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
    for (int w = 0; w < nw; w++) tot += red[w];
    scale = 1.0f / sqrtf(tot / (float)H + 1e-6f);
    __syncthreads();
  }
  float gdot = 0.f;
  for (int i = threadIdx.x; i < H; i += blockDim.x) {
    const float v = xr[i] * scale;
    const uint32_t hi = f2bf_rn(v);
    const uint32_t lo = f2bf_rn(v - __uint_as_float(hi << 16));
    P.xr_hi[(size_t)tok * H + i] = (uint16_t)hi;
    P.xr_lo[(size_t)tok * H + i] = (uint16_t)lo;
    P.xg[(size_t)tok * H + (i & ~7) + perm8(i & 7)] = (uint16_t)hi;
    if (P.sgate) gdot += __uint_as_float((uint32_t)P.sgate[i] << 16) * v;
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
// blockIdx.x + gridDim.x, ... of a 128 x N (N <= 256) output tile list; K
// goes in stages of 64 through a ring of kS shared-memory stages.
//   warp 0      lane 0 issues the tcgen05 MMAs of a stage once its operands
//               have landed and commits them (stage free / accumulator full)
//   warp 1      TMA: B rows (and the router's A rows) of each stage
//   warps 2-9   A producers, two groups of four warps taking alternate
//               stages: thread r of a group dequantizes weight row r of the
//               tile (64 codes = one group per stage) to bf16 in the
//               swizzled layout; each group's loads run four of its stages
//               (eight stages in all) ahead, enough bytes in flight to
//               stream the codes at HBM rate
//   warps 10-13 epilogue: TMEM -> registers -> global, from one of two
//               accumulators while the MMAs fill the other
// Every mbarrier wait is bounded; a wait that gives up records
// MOE_ETIMEOUT in *status and its role stops, so the CTA ends.

constexpr int kWsThreads = 320;
constexpr int kS = 3;                      // A / B pipeline stages
constexpr int kChunk = 4;                  // k-stages per staged chunk of codes
constexpr int kStgCodes = 128 * 128;       // 128 rows x 128 bytes of codes (4 stages)
constexpr int kStgSB = 128 * kChunk * 8;   // per row and stage: scale word, bias word
constexpr int kStgBuf = kStgCodes + kStgSB;
constexpr int kNStg = 3;                   // staged chunks: one being read, two in flight
constexpr int kOffB = kS * kStageA;        // B stages follow the A stages
constexpr int kOffStg = kOffB + kS * kStageB;
constexpr int kOffEpi = kOffStg + kNStg * kStgBuf;
constexpr int kEpiBytes = 16384;           // down: 4 warps x 32 x 32 fp32; gate_up: exchange + h rows
constexpr int kOffTile = kOffEpi + kEpiBytes;
constexpr int kOffBars = kOffTile + 2 * kPfTileN * 4;
constexpr int kWsSmem = kOffBars + 256 + 1024;  // + alignment slack
static_assert(kWsSmem <= 227 * 1024, "shared memory");

struct WsBars {
  uint64_t full_b[kS], full_a[kS], empty[kS], acc_full[2], acc_empty[2], drain;
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

// Weight row `r` of a tile: gate_up tiles hold 64 gate rows then the 64
// matching up rows; down tiles 128 output rows.
template <int MODE>
__device__ __forceinline__ int ws_weight_row(const PfParams &P, int mt, int r) {
  if constexpr (MODE == MODE_GATE_UP)
    return r < 64 ? mt * 64 + r : P.I + mt * 64 + (r - 64);
  else
    return mt * 128 + r;
}

// Stage one chunk of codes (k-stages 4kc .. 4kc+3 of a tile) into shared
// memory: 128 rows x 128 bytes, copied by 8 threads per row segment so that
// each warp instruction reads four whole 128-byte lines (16-byte pieces
// placed at piece ^ (row & 7) against bank conflicts); plus, per row and
// stage, the 4-byte words holding its scale and bias.  A segment may run
// past the end of a row, into bytes of the same record (codes are followed
// by the scale and bias tables); those bytes are never used.
template <int MODE>
__device__ __forceinline__ void stage_chunk(const PfParams &P, const PfItem &it, int kc, int nk, int r, uint8_t *buf) {
  if (item_ok<MODE>(it)) {
    const uint8_t *rec = reinterpret_cast<const uint8_t *>(it.rec);
    const QOff q = it.g == P.E ? (MODE == MODE_GATE_UP ? P.sgu : P.sdn) : (MODE == MODE_GATE_UP ? P.gu : P.dn);
    const int inp = MODE == MODE_GATE_UP ? P.H : P.I;
#pragma unroll
    for (int i = 0; i < 8; i++) {
      const int idx = i * 128 + r, row = idx >> 3, part = idx & 7;
      const size_t src = q.w + (size_t)ws_weight_row<MODE>(P, it.mt, row) * (inp / 2) + kc * 128 + part * 16;
      tc05::cp16(buf + row * 128 + ((part ^ (row & 7)) << 4), rec + src);
    }
    const size_t gbase = (size_t)ws_weight_row<MODE>(P, it.mt, r) * (inp / 64);
#pragma unroll
    for (int u = 0; u < kChunk; u++) {
      const int kk = min(kc * kChunk + u, nk - 1);
      const size_t gi = (gbase + kk) * 2;
      tc05::cp4(buf + kStgCodes + (r * kChunk + u) * 8, rec + ((q.s + gi) & ~(size_t)3));
      tc05::cp4(buf + kStgCodes + (r * kChunk + u) * 8 + 4, rec + ((q.b + gi) & ~(size_t)3));
    }
  }
  tc05::cp_commit();
}

// 64 codes of row r, stage u of a staged chunk -> bf16(scale * code + bias),
// k permuted within 8-blocks, into row r of a swizzled A stage
__device__ __forceinline__ void ws_dequant_row(const uint8_t *buf, int r, int u, uint32_t half, uint8_t *sA) {
  const uint8_t *row = buf + r * 128;
  const uint4 c0 = *reinterpret_cast<const uint4 *>(row + (((2 * u) ^ (r & 7)) << 4));
  const uint4 c1 = *reinterpret_cast<const uint4 *>(row + (((2 * u + 1) ^ (r & 7)) << 4));
  const uint2 sbw = *reinterpret_cast<const uint2 *>(buf + kStgCodes + (r * kChunk + u) * 8);
  const uint32_t s = (sbw.x >> (16 * half)) & 0xffffu, b = (sbw.y >> (16 * half)) & 0xffffu;
  const uint32_t s2 = s * 0x10001u, b2 = b * 0x10001u;
  const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
  for (int ch = 0; ch < 8; ch++) {
    uint32_t pr[4];
#pragma unroll
    for (int j = 0; j < 4; j++) {
      const uint32_t v = ((w[ch] >> (4 * j)) & 0x000f000fu) | 0x43004300u;  // (128 + n_j, 128 + n_{j+4})
      const uint32_t qv = bfma2(v, 0x3f803f80u, 0xc300c300u);              // the codes, exact
      pr[j] = bfma2(qv, s2, b2);                                            // bf16(s*q + b)
    }
    *reinterpret_cast<uint4 *>(sA + tc05::sw128_offset(r, ch)) = make_uint4(pr[0], pr[1], pr[2], pr[3]);
  }
}

template <int MODE>
__global__ void __launch_bounds__(kWsThreads, 1) pf_gemm(const __grid_constant__ PfParams P) {
  extern __shared__ __align__(1024) uint8_t smraw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~(uintptr_t)1023);
  WsBars &B = *reinterpret_cast<WsBars *>(sm + kOffBars);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ntiles = ws_num_tiles<MODE>(P);
  const int nk = ws_nk<MODE>(P);
  const int my_tiles = (int)blockIdx.x < ntiles ? (ntiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  auto tile_of = [&](int lt) { return (int)blockIdx.x + lt * (int)gridDim.x; };

  if (tid == 0) {
    for (int s = 0; s < kS; s++) {
      mbar_init(&B.full_b[s], 1);
      mbar_init(&B.full_a[s], 4);
      mbar_init(&B.empty[s], 1);
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

  if (warp == 0) {
    // ---------------------------------------------------------------- MMA issue
    if (lane == 0) {
      int f = 0;
      bool ok = true;
      PfItem nx{};
      if (my_tiles > 0) nx = ws_item<MODE>(P, tile_of(0));
      for (int lt = 0; lt < my_tiles && ok; lt++) {
        const PfItem cur = nx;
        if (lt + 1 < my_tiles) nx = ws_item<MODE>(P, tile_of(lt + 1));
        const int b = lt & 1;
        if (!pf_wait(&B.acc_empty[b], (uint32_t)(((lt >> 1) & 1) ^ 1), P)) {
          ok = false;
          break;
        }
        tc05::fence_after();
        const uint32_t d = tmem + (uint32_t)(b * 256);
        const uint32_t idesc = tc05::idesc_bf16(tile_n(cur));
        for (int kk = 0; kk < nk; kk++, f++) {
          const int s = f % kS;
          const uint32_t par = (uint32_t)((f / kS) & 1);
          if (!pf_wait(&B.full_b[s], par, P) || (MODE != MODE_ROUTER && !pf_wait(&B.full_a[s], par, P))) {
            ok = false;
            break;
          }
          tc05::fence_after();
          const uint32_t a0 = smem_u32(sm + s * kStageA), b0 = smem_u32(sm + kOffB + s * kStageB);
#pragma unroll
          for (int j = 0; j < 4; j++)
            tc05::mma(d, tc05::sdesc(a0 + 32 * j), tc05::sdesc(b0 + 32 * j), idesc, (kk | j) != 0);
          tc05::commit(&B.empty[s]);
        }
        if (ok) tc05::commit(&B.acc_full[b]);
      }
      // every MMA issued here has completed before TMEM is released
      tc05::commit(&B.drain);
      pf_wait(&B.drain, 0, P);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- B producer (TMA)
    // router: 128 token rows of x^ hi / lo and the 128 router rows; gate_up
    // and down: the tile's rows of the grouped operand (x^ rows gathered in
    // group order, or h), boxes of 128 rows then 32-row boxes for the tail
    int f = 0;
    PfItem ia{}, ib{};
    if (my_tiles > 0) ia = ws_item<MODE>(P, tile_of(0));
    bool ok = true;
    for (int lt = 0; lt < my_tiles && ok; lt++) {
      if (lt + 1 < my_tiles) ib = ws_item<MODE>(P, tile_of(lt + 1));
      const int N = tile_n(ia);
      const int n128 = N >> 7, n32 = ((N & 127) + 31) >> 5;
      const uint32_t bytes = MODE == MODE_ROUTER ? (uint32_t)(kStageA + 128 * 128)
                                                 : (uint32_t)(n128 * 128 + n32 * 32) * 128u;
      const CUtensorMap *m128 = MODE == MODE_GATE_UP ? &P.tm_xc : &P.tm_h;
      const CUtensorMap *m32 = MODE == MODE_GATE_UP ? &P.tm_xc32 : &P.tm_h32;
      for (int kk = 0; kk < nk; kk++, f++) {
        const int s = f % kS;
        if (!warp_wait(&B.empty[s], (uint32_t)(((f / kS) & 1) ^ 1), P)) {
          ok = false;
          break;
        }
        uint8_t *sb = sm + kOffB + s * kStageB;
        if (lane == 0) mbar_expect_tx(&B.full_b[s], bytes);
        __syncwarp();
        if constexpr (MODE == MODE_ROUTER) {
          const int nq = P.H / 64, kq = kk % nq, yb = (kk < nq ? 0 : P.t) + ia.n0;
          if (lane == 0) {
            tc05::tma_load_2d(sm + s * kStageA, &P.tm_router, kq * 64, ia.mt * 128, &B.full_b[s]);
            tc05::tma_load_2d(sb, &P.tm_xr, kq * 64, yb, &B.full_b[s]);
          }
        } else {
          if (lane < n128) tc05::tma_load_2d(sb + lane * 128 * 128, m128, kk * 64, ia.n0 + lane * 128, &B.full_b[s]);
          if (lane < n32)
            tc05::tma_load_2d(sb + (n128 * 128 + lane * 32) * 128, m32, kk * 64, ia.n0 + n128 * 128 + lane * 32,
                              &B.full_b[s]);
        }
      }
      ia = ib;
    }
    // copies still in flight land before the CTA ends
    if (lane == 0 && f > 0) pf_wait(&B.full_b[(f - 1) % kS], (uint32_t)(((f - 1) / kS) & 1), P);
    __syncwarp();
  } else if (warp < 6) {
    // ---------------------------------------------------------------- A producers
    if constexpr (MODE != MODE_ROUTER) {
      const int r = tid - 64;
      const int nct = (nk + kChunk - 1) / kChunk;  // chunks per tile
      const int total = my_tiles * nct;
      const int inp = MODE == MODE_GATE_UP ? P.H : P.I;
      uint8_t *stg = sm + kOffStg;
      // items of the staging position's tile and of the tile after it
      PfItem scur{}, snext{};
      int slt = 0;
      if (my_tiles > 0) scur = ws_item<MODE>(P, tile_of(0));
      if (my_tiles > 1) snext = ws_item<MODE>(P, tile_of(1));
      auto issue = [&](int c) {
        if (c >= total) {
          tc05::cp_commit();  // empty group keeps the group count uniform
          return;
        }
        const int lt = c / nct;
        if (lt != slt) {
          scur = lt == slt + 1 ? snext : ws_item<MODE>(P, tile_of(lt));
          slt = lt;
          if (lt + 1 < my_tiles) snext = ws_item<MODE>(P, tile_of(lt + 1));
        }
        stage_chunk<MODE>(P, scur, c - lt * nct, nk, r, stg + (c % kNStg) * kStgBuf);
      };
      issue(0);
      issue(1);
      // parity of the weight row = parity of r (tile row bases are even)
      const uint32_t rodd = (uint32_t)(r & (inp / 64) & 1);
      bool ok = true;
      for (int c = 0; c < total && ok; c++) {
        tc05::cp_wait_group<1>();  // this thread's copies of chunk c are done
        tc05::named_sync(3, 128);  // everyone's are; everyone is done reading chunk c - 1
        issue(c + 2);
        const int lt = c / nct, kc = c - lt * nct;
        const uint8_t *buf = stg + (c % kNStg) * kStgBuf;
        const int ns = min(kChunk, nk - kc * kChunk);
        for (int u = 0; u < ns; u++) {
          const int kk = kc * kChunk + u, f = lt * nk + kk, s = f % kS;
          if (!warp_wait(&B.empty[s], (uint32_t)(((f / kS) & 1) ^ 1), P)) {
            ok = false;
            break;
          }
          // scale / bias: the half of the staged 4-byte word holding entry row * G + kk
          const uint32_t half = (rodd + (uint32_t)kk) & 1u;
          ws_dequant_row(buf, r, u, half, sm + s * kStageA);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) tc05::mbar_arrive(&B.full_a[s]);
        }
        // the four producer warps stop together (they share a named barrier)
        ok = tc05::named_and(4, 128, ok);
      }
      tc05::cp_wait_group<0>();  // nothing in flight into shared memory at the end
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;    // TMEM lane quadrant this warp may read
    const int et = tid - 192;  // 0..127 over the epilogue warps
    int *trow = reinterpret_cast<int *>(sm + kOffTile);
    float *twt = reinterpret_cast<float *>(sm + kOffTile) + kPfTileN;
    PfItem nx{};
    int pr[2] = {0, 0};
    float pw[2] = {0.f, 0.f};
    auto fetch_entries = [&](const PfItem &it) {  // down: this thread's two entries of a tile
#pragma unroll
      for (int h = 0; h < 2; h++) {
        const int j = et + 128 * h;
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
        for (int h = 0; h < 2; h++) trow[et + 128 * h] = pr[h], twt[et + 128 * h] = pw[h];
        tc05::named_sync(1, 128);
      }
      // the four epilogue warps stop together (they share named barriers)
      if (!tc05::named_and(2, 128, warp_wait(&B.acc_full[b], (uint32_t)((lt >> 1) & 1), P))) break;
      tc05::fence_after();
      const uint32_t tl = tmem + (uint32_t)(b * 256) + ((uint32_t)(32 * q) << 16);
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
            float *tb = reinterpret_cast<float *>(sm + kOffEpi) + (warp - 6) * 1024;
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
            // up rows (quadrants 2, 3) -> shared; h = silu(gate) * up on quadrants 0, 1
            float *xch = reinterpret_cast<float *>(sm + kOffEpi);
            uint16_t *hs = reinterpret_cast<uint16_t *>(xch + 64 * 33);  // [32 tokens][64] bf16, permuted k
            tc05::named_sync(1, 128);
            if (q >= 2)
#pragma unroll
              for (int j = 0; j < 32; j++) xch[(32 * (q - 2) + lane) * 33 + j] = v[j];
            tc05::named_sync(1, 128);
            if (q < 2) {
              const int i = 32 * q + lane;
#pragma unroll
              for (int j = 0; j < 32; j++) {
                const float g = v[j], u = xch[i * 33 + j];
                const float h = g / (1.f + expf(-g)) * u;
                hs[j * 64 + (i & ~7) + perm8(i & 7)] = (uint16_t)f2bf_rn(h);
              }
            }
            tc05::named_sync(1, 128);
            for (int i = et; i < 32 * 8; i += 128) {
              const int j = i >> 3, c = i & 7;
              if (c0 + j < T.nlen)
                *reinterpret_cast<uint4 *>(P.hbuf + (size_t)(T.n0 + c0 + j) * P.I + T.mt * 64 + c * 8) =
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

// Expert operand rows in group order: xc[e] = x^ row of grouped entry e
// (warp per entry, 16-byte copies), so that the gate_up GEMM reads its
// token rows as plain TMA boxes.
__global__ void pf_gather(const __grid_constant__ PfParams P) {
  const int e = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  const int G = P.E + (P.sgate ? 1 : 0);
  if (e >= P.offs[G]) return;
  const uint4 *src = reinterpret_cast<const uint4 *>(P.xg + (size_t)P.rows[e] * P.H);
  uint4 *dst = reinterpret_cast<uint4 *>(P.xc + (size_t)e * P.H);
  for (int i = lane; i < P.H / 8; i += 32) dst[i] = src[i];
}

// ------------------------------------------------------------ routing

__device__ __forceinline__ uint32_t orderable_f(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Warp per token: top-k (ties to the lower id) of E <= 1024 logits, softmax
// over the k chosen, per-(chunk, expert) counts.
__global__ void pf_topk(const __grid_constant__ PfParams P) {
  const int lane = threadIdx.x & 31;
  const int tok = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (tok >= P.t) return;
  const int E = P.E, K = P.K, PP = (E + 31) / 32;
  const float *lg = P.logits + (size_t)tok * E;
  uint32_t key[32];
#pragma unroll
  for (int i = 0; i < 32; i++) {
    const int e = lane * PP + i;
    key[i] = (i < PP && e < E) ? orderable_f(lg[e]) : 0u;
  }
  uint32_t bk = 0;
  int bi = 0;
#pragma unroll
  for (int i = 0; i < 32; i++)
    if (key[i] > bk) bk = key[i], bi = i;
  float myl = 0.f;
  int myid = 0;
  for (int r = 0; r < K; r++) {
    const uint32_t m = __reduce_max_sync(FULLM, bk);
    const int wl = __ffs(__ballot_sync(FULLM, bk == m)) - 1;
    const int id = __shfl_sync(FULLM, lane * PP + bi, wl);
    if (lane == r) myid = id, myl = lg[id];
    if (lane == wl) {
      uint32_t nbk = 0;
      int nbi = 0;
#pragma unroll
      for (int i = 0; i < 32; i++) {
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
    atomicAdd(&P.chist[(tok / kPfChunk) * E + myid], 1);
  }
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

// One block of 1024 threads: groups g = 2i, 2i+1 per thread (experts, then
// the shared expert with all tokens): offsets, per-chunk list bases, tile
// work lists.
__global__ void __launch_bounds__(1024) pf_group(const __grid_constant__ PfParams P) {
  __shared__ int sh[32];
  const int E = P.E, G = E + (P.sgate ? 1 : 0), nch = (P.t + kPfChunk - 1) / kPfChunk;
  const int nmt1 = P.I / 64, nmt2 = P.H / 128;
  int m[2], ch[2];
#pragma unroll
  for (int u = 0; u < 2; u++) {
    const int g = 2 * threadIdx.x + u;
    int c = 0;
    if (g < E)
      for (int k = 0; k < nch; k++) c += P.chist[k * E + g];
    else if (g < G)
      c = P.t;
    m[u] = c;
    ch[u] = (c + kPfTileN - 1) / kPfTileN;
  }
  int tot_m, tot_ch;
  const int om = block_exscan(m[0] + m[1], sh, &tot_m);
  const int oc = block_exscan(ch[0] + ch[1], sh, &tot_ch);
  const int offs[2] = {om, om + m[0]}, ocs[2] = {oc, oc + ch[0]};
#pragma unroll
  for (int u = 0; u < 2; u++) {
    const int g = 2 * threadIdx.x + u;
    if (g < G) {
      P.offs[g] = offs[u];
      if (g < E) {  // chunk bases: ascending chunks keep ascending tokens
        int b = offs[u];
        for (int k = 0; k < nch; k++) {
          const int c = P.chist[k * E + g];
          P.chist[k * E + g] = b;
          b += c;
        }
      }
      const uint64_t rec = g < E ? P.eaddr[g] : reinterpret_cast<uint64_t>(P.srec);
      int a = ocs[u] * nmt1, bb = ocs[u] * nmt2;
      for (int c = 0; c < ch[u]; c++) {
        const int n0 = offs[u] + c * kPfTileN, nl = min(kPfTileN, m[u] - c * kPfTileN);
        for (int mt = 0; mt < nmt1; mt++) P.items1[a++] = PfItem{g, mt, n0, nl, rec};
        for (int mt = 0; mt < nmt2; mt++) P.items2[bb++] = PfItem{g, mt, n0, nl, rec};
      }
    }
  }
  if (threadIdx.x == 0) {
    P.offs[G] = tot_m;
    P.nitems[0] = tot_ch * nmt1, P.nitems[1] = tot_ch * nmt2;
  }
}

// One warp per chunk of kPfChunk tokens: the chunk's (token, expert) pairs in
// token order get consecutive places in their experts' lists, so every list
// is in ascending token order.  Shared group: every token, weight = gate.
__global__ void pf_fill(const __grid_constant__ PfParams P) {
  extern __shared__ int cnt[];  // [E] next place of each expert for this chunk
  const int E = P.E, K = P.K, c = blockIdx.x, lane = threadIdx.x;
  for (int e = lane; e < E; e += 32) cnt[e] = P.chist[c * E + e];
  __syncwarp();
  const int t0 = c * kPfChunk, t1 = min(P.t, t0 + kPfChunk);
  for (int i0 = t0 * K; i0 < t1 * K; i0 += 32) {
    const int i = i0 + lane;
    const bool v = i < t1 * K;
    const int e = v ? P.tk_idx[i] : -1;
    const unsigned peers = __match_any_sync(FULLM, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const int base = v ? cnt[e] : 0;
    __syncwarp();
    if (v) {
      P.rows[base + rank] = i / K;
      P.wts[base + rank] = P.tk_w[i];
      if (rank == 0) cnt[e] = base + __popc(peers);
    }
    __syncwarp();
  }
  if (P.sgate) {
    const int o = P.offs[E];
    for (int tok = t0 + lane; tok < t1; tok += 32) {
      P.rows[o + tok] = tok;
      P.wts[o + tok] = P.gam[tok];
    }
  }
}

__global__ void pf_final(const __grid_constant__ PfParams P) {
  const size_t n = (size_t)P.t * P.H;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    float y = P.Y[i];
    if (P.flags & kResidualF) y += P.x[i];
    P.out[i] = (uint16_t)f2bf_rn(y);
  }
}

size_t al(size_t n) { return (n + 1023) & ~(size_t)1023; }

// upper bound of the work items of one GEMM: sum over groups of
// ceil(m_g / 256) <= entries / 256 + groups
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
  take(9, ent * 4);              // rows
  take(10, ent * 4);             // wts
  take(11, items * (I / 64) * sizeof(PfItem));
  take(12, items * (H / 128) * sizeof(PfItem));
  take(13, 64);                  // nitems
  take(14, ent * I * 2);         // hbuf
  take(15, (size_t)t * H * 4);   // Y
  take(16, ent * H * 2);         // xc
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
  void *ptr[17];
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
      !make_map(&p.tm_h, p.hbuf, (uint64_t)p.I, ent, 128) || !make_map(&p.tm_h32, p.hbuf, (uint64_t)p.I, ent, 32) ||
      !make_map(&p.tm_xc, p.xc, H, ent, 128) || !make_map(&p.tm_xc32, p.xc, H, ent, 32)) {
    *why = "cuTensorMapEncodeTiled rejected a tensor map";
    return -1;
  }
  return 0;
}

cudaError_t pf_launch(PfParams &p, cudaStream_t st, cudaEvent_t const *events) {
  const int t = p.t, nch = (t + kPfChunk - 1) / kPfChunk;
  const size_t ent_cap = (size_t)t * (p.K + 1);
  cudaError_t e;
  auto mark = [&](int i) { return events ? cudaEventRecord(events[i], st) : cudaSuccess; };
  if ((e = cudaMemsetAsync(p.chist, 0, (size_t)nch * p.E * 4, st))) return e;
  if ((e = cudaMemsetAsync(p.status, 0, 4, st))) return e;
  if (!p.route_only && (e = cudaMemsetAsync(p.Y, 0, (size_t)t * p.H * 4, st))) return e;
  if ((e = cudaFuncSetAttribute(pf_gemm<MODE_ROUTER>, cudaFuncAttributeMaxDynamicSharedMemorySize, kWsSmem)))
    return e;
  if ((e = cudaFuncSetAttribute(pf_gemm<MODE_GATE_UP>, cudaFuncAttributeMaxDynamicSharedMemorySize, kWsSmem)))
    return e;
  if ((e = cudaFuncSetAttribute(pf_gemm<MODE_DOWN>, cudaFuncAttributeMaxDynamicSharedMemorySize, kWsSmem))) return e;
  const int ntr = ((p.E + 127) / 128) * ((t + 127) / 128);
  const int g_router = ntr < p.n_sms ? ntr : p.n_sms;
  if ((e = mark(0))) return e;
  pf_prep<<<t, 256, 0, st>>>(p);
  if ((e = mark(1))) return e;
  pf_gemm<MODE_ROUTER><<<g_router, kWsThreads, kWsSmem, st>>>(p);
  if ((e = mark(2))) return e;
  pf_topk<<<(t + 7) / 8, 256, 0, st>>>(p);
  if ((e = mark(3))) return e;
  pf_group<<<1, 1024, 0, st>>>(p);
  if ((e = mark(4))) return e;
  pf_fill<<<nch, 32, (size_t)p.E * 4, st>>>(p);
  if ((e = mark(5))) return e;
  if (!p.route_only) {
    pf_gather<<<(int)((ent_cap + 7) / 8), 256, 0, st>>>(p);
    if ((e = mark(6))) return e;
    pf_gemm<MODE_GATE_UP><<<p.n_sms, kWsThreads, kWsSmem, st>>>(p);
    if ((e = mark(7))) return e;
    pf_gemm<MODE_DOWN><<<p.n_sms, kWsThreads, kWsSmem, st>>>(p);
    if ((e = mark(8))) return e;
    pf_final<<<1024, 256, 0, st>>>(p);
    if ((e = mark(9))) return e;
  }
  return cudaGetLastError();
}

}  // namespace moe
