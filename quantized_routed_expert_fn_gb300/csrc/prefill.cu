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

constexpr int PT = 128;  // threads of a tensor-core CTA (one warpgroup)
constexpr unsigned FULLM = 0xffffffffu;
constexpr uint32_t kResidualF = 1, kPrenormF = 2;
enum { MODE_ROUTER = 0, MODE_GATE_UP = 1, MODE_DOWN = 2 };

constexpr int kStageA = 128 * 128;       // 128 rows x 64 k bf16
constexpr int kStageB = kPfTileN * 128;  // 256 rows x 64 k bf16
constexpr int kSmem = 2 * kStageA + 2 * kStageB + 64 + 1024;

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
// One CTA (one warpgroup) computes a 128 x N tile, N <= 256, over all K in
// stages of 64: thread r writes row r of A (dequantized or copied), the
// token rows of B arrive by cp.async, thread 0 issues four k=16 MMAs per
// stage and commits them to the stage's mbarrier; two stages alternate.

// A rows of one stage.  Row r of the tile, k range [64*kk, 64*kk + 64).
template <int MODE>
__device__ __forceinline__ void produce_a(const PfParams &P, const PfItem &it, const uint8_t *rec, const QOff &q,
                                          int kk, uint8_t *sA) {
  const int r = threadIdx.x;
  if constexpr (MODE == MODE_ROUTER) {
    const int H = P.H, e = it.mt * 128 + r;
    const int kq = kk % (H / 64);
    if (e < P.E) {
      const uint8_t *src = reinterpret_cast<const uint8_t *>(P.router + (size_t)e * H + kq * 64);
#pragma unroll
      for (int c = 0; c < 8; c++) tc05::cp16(sA + tc05::sw128_offset(r, c), src + c * 16);
    } else {
#pragma unroll
      for (int c = 0; c < 8; c++) *reinterpret_cast<uint4 *>(sA + tc05::sw128_offset(r, c)) = make_uint4(0, 0, 0, 0);
    }
  } else {
    // 4-bit affine row of 64 codes = one group: W = scale * code + bias in
    // bf16 (exact product and sum, one rounding), k permuted within 8-blocks
    const int inp = MODE == MODE_GATE_UP ? P.H : P.I;
    int row;
    if (MODE == MODE_GATE_UP)
      row = r < 64 ? it.mt * 64 + r : P.I + it.mt * 64 + (r - 64);
    else
      row = it.mt * 128 + r;
    const uint8_t *cp = rec + q.w + (size_t)row * (inp / 2) + kk * 32;
    const uint4 w0 = *reinterpret_cast<const uint4 *>(cp);
    const uint4 w1 = *reinterpret_cast<const uint4 *>(cp + 16);
    const uint32_t s = *reinterpret_cast<const uint16_t *>(rec + q.s + ((size_t)row * (inp / 64) + kk) * 2);
    const uint32_t b = *reinterpret_cast<const uint16_t *>(rec + q.b + ((size_t)row * (inp / 64) + kk) * 2);
    const uint32_t s2 = s | (s << 16), b2 = b | (b << 16);
    const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
    for (int c = 0; c < 8; c++) {
      uint32_t pr[4];
#pragma unroll
      for (int j = 0; j < 4; j++) {
        const uint32_t v = ((w[c] >> (4 * j)) & 0x000f000fu) | 0x43004300u;  // (128 + n_j, 128 + n_{j+4})
        const uint32_t qv = bfma2(v, 0x3f803f80u, 0xc300c300u);             // the codes, exact
        pr[j] = bfma2(qv, s2, b2);                                           // bf16(s*q + b)
      }
      *reinterpret_cast<uint4 *>(sA + tc05::sw128_offset(r, c)) = make_uint4(pr[0], pr[1], pr[2], pr[3]);
    }
  }
}

// B rows of one stage: token rows [0, N); rows >= nlen are zero.
template <int MODE>
__device__ __forceinline__ void produce_b(const PfParams &P, const PfItem &it, int N, int kk, uint8_t *sB) {
  for (int i = threadIdx.x; i < N * 8; i += PT) {
    const int j = i >> 3, c = i & 7;
    uint8_t *dst = sB + tc05::sw128_offset(j, c);
    if (j < it.nlen) {
      const uint8_t *src;
      if constexpr (MODE == MODE_ROUTER) {
        const int nq = P.H / 64;
        const uint16_t *base = kk < nq ? P.xr_hi : P.xr_lo;
        src = reinterpret_cast<const uint8_t *>(base + (size_t)(it.n0 + j) * P.H + (kk % nq) * 64);
      } else if constexpr (MODE == MODE_GATE_UP) {
        src = reinterpret_cast<const uint8_t *>(P.xg + (size_t)P.rows[it.n0 + j] * P.H + kk * 64);
      } else {
        src = reinterpret_cast<const uint8_t *>(P.hbuf + (size_t)(it.n0 + j) * P.I + kk * 64);
      }
      tc05::cp16(dst, src + c * 16);
    } else {
      *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
    }
  }
}

template <int MODE>
__global__ void __launch_bounds__(PT) pf_gemm(const __grid_constant__ PfParams P) {
  extern __shared__ __align__(1024) uint8_t smraw[];
  // the swizzled tiles want 1024-byte alignment
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~(uintptr_t)1023);
  uint8_t *sA = sm, *sB = sm + 2 * kStageA;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + 2 * kStageA + 2 * kStageB);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + 2);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  PfItem it;
  if constexpr (MODE == MODE_ROUTER) {
    const int nmt = (P.E + 127) / 128;
    it.g = 0, it.mt = blockIdx.x % nmt, it.n0 = (blockIdx.x / nmt) * 128;
    it.nlen = min(128, P.t - it.n0);
  } else {
    const int n = P.nitems[MODE == MODE_GATE_UP ? 0 : 1];
    if ((int)blockIdx.x >= n) return;
    it = (MODE == MODE_GATE_UP ? P.items1 : P.items2)[blockIdx.x];
  }
  const int N = (it.nlen + 15) & ~15;
  const uint8_t *rec = nullptr;
  QOff q = {0, 0, 0};
  if constexpr (MODE != MODE_ROUTER) {
    const bool shared = it.g == P.E;
    rec = shared ? P.srec : reinterpret_cast<const uint8_t *>(P.eaddr[it.g]);
    q = shared ? (MODE == MODE_GATE_UP ? P.sgu : P.sdn) : (MODE == MODE_GATE_UP ? P.gu : P.dn);
    if (rec == nullptr || ((uintptr_t)rec & 15u)) {
      if (tid == 0) atomicCAS(P.status, 0, kStatusDevice);
      return;
    }
  }
  const int nk = MODE == MODE_ROUTER ? 2 * P.H / 64 : (MODE == MODE_GATE_UP ? P.H / 64 : P.I / 64);

  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
  if (warp == 0) tc05::alloc(tslot, 256);
  tc05::fence_before();
  __syncthreads();
  tc05::fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t idesc = tc05::idesc_bf16(N);

  bool ok = true;
  int kk = 0;
  for (; kk < nk; kk++) {
    const int s = kk & 1;
    // the MMAs that read this stage two steps ago are done
    if (kk >= 2 && !__syncthreads_and(pf_wait(&bars[s], (uint32_t)(((kk - 2) >> 1) & 1), P))) {
      ok = false;
      break;
    }
    produce_a<MODE>(P, it, rec, q, kk, sA + s * kStageA);
    produce_b<MODE>(P, it, N, kk, sB + s * kStageB);
    tc05::cp_wait_all();
    fence_proxy_async_smem();  // generic-proxy shared writes -> visible to the tensor core
    __syncthreads();
    if (tid == 0) {
      tc05::fence_after();
      const uint32_t a0 = smem_u32(sA + s * kStageA), b0 = smem_u32(sB + s * kStageB);
#pragma unroll
      for (int j = 0; j < 4; j++)
        tc05::mma(tmem, tc05::sdesc(a0 + 32 * j), tc05::sdesc(b0 + 32 * j), idesc, (kk | j) != 0);
      tc05::commit(&bars[s]);
    }
  }
  // the last commit covers every MMA issued before it
  if (kk > 0 && !__syncthreads_and(pf_wait(&bars[(kk - 1) & 1], (uint32_t)(((kk - 1) >> 1) & 1), P))) ok = false;
  tc05::fence_after();

  if (ok) {
    // ---- epilogue: warp w owns TMEM lanes (tile rows) 32w .. 32w+31
    const uint32_t tl = tmem + ((uint32_t)(32 * warp) << 16);
    float *xch = reinterpret_cast<float *>(sm);  // reuses the stages
    for (int c0 = 0; c0 < N; c0 += 32) {
      float v[32];
      tc05::ld32(tl + c0, v);
      if constexpr (MODE == MODE_ROUTER) {
        const int e = it.mt * 128 + 32 * warp + lane;
        if (e < P.E)
#pragma unroll
          for (int j = 0; j < 32; j++)
            if (c0 + j < it.nlen) P.logits[(size_t)(it.n0 + c0 + j) * P.E + e] = v[j];
      } else if constexpr (MODE == MODE_DOWN) {
        const int o = it.mt * 128 + 32 * warp + lane;
#pragma unroll
        for (int j = 0; j < 32; j++) {
          if (c0 + j < it.nlen) {
            const int ent = it.n0 + c0 + j;
            atomicAdd(&P.Y[(size_t)P.rows[ent] * P.H + o], P.wts[ent] * v[j]);
          }
        }
      } else {
        // up rows (lanes 64..127) -> shared, then h = silu(gate) * up on lanes 0..63
        __syncthreads();
        if (warp >= 2)
#pragma unroll
          for (int j = 0; j < 32; j++) xch[(32 * (warp - 2) + lane) * 33 + j] = v[j];
        __syncthreads();
        uint16_t *hs = reinterpret_cast<uint16_t *>(xch + 64 * 33);  // [32 tokens][64] bf16, permuted k
        if (warp < 2) {
          const int i = 32 * warp + lane;  // gate row inside the tile
#pragma unroll
          for (int j = 0; j < 32; j++) {
            const float g = v[j], u = xch[i * 33 + j];
            const float h = g / (1.f + expf(-g)) * u;
            hs[j * 64 + (i & ~7) + perm8(i & 7)] = (uint16_t)f2bf_rn(h);
          }
        }
        __syncthreads();
        // 32 tokens x 128 bytes -> hbuf rows (k = mt*64 .. +64)
        for (int i = tid; i < 32 * 8; i += PT) {
          const int j = i >> 3, c = i & 7;
          if (c0 + j < it.nlen)
            *reinterpret_cast<uint4 *>(P.hbuf + (size_t)(it.n0 + c0 + j) * P.I + it.mt * 64 + c * 8) =
                *reinterpret_cast<const uint4 *>(hs + j * 64 + c * 8);
        }
      }
    }
  }
  tc05::fence_before();
  __syncthreads();
  if (warp == 0) tc05::dealloc(tmem, 256);
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
      int a = ocs[u] * nmt1, bb = ocs[u] * nmt2;
      for (int c = 0; c < ch[u]; c++) {
        const int n0 = offs[u] + c * kPfTileN, nl = min(kPfTileN, m[u] - c * kPfTileN);
        for (int mt = 0; mt < nmt1; mt++) P.items1[a++] = PfItem{g, mt, n0, nl};
        for (int mt = 0; mt < nmt2; mt++) P.items2[bb++] = PfItem{g, mt, n0, nl};
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
  take(0, (size_t)t * H * 2);    // xr_hi
  take(1, (size_t)t * H * 2);    // xr_lo
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
  void *ptr[16];
  carve(p.H, p.E, p.K, p.I, p.t, [&](int k, size_t n) {
    ptr[k] = base + o;
    o += al(n);
  });
  p.xr_hi = (uint16_t *)ptr[0];
  p.xr_lo = (uint16_t *)ptr[1];
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
}

cudaError_t pf_launch(PfParams &p, cudaStream_t st) {
  const int t = p.t, nch = (t + kPfChunk - 1) / kPfChunk;
  const int items = (int)max_items(p.E, p.K, t);
  cudaError_t e;
  if ((e = cudaMemsetAsync(p.chist, 0, (size_t)nch * p.E * 4, st))) return e;
  if ((e = cudaMemsetAsync(p.status, 0, 4, st))) return e;
  static_assert(kSmem <= 227 * 1024, "shared memory");
  if ((e = cudaFuncSetAttribute(pf_gemm<MODE_ROUTER>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem))) return e;
  if ((e = cudaFuncSetAttribute(pf_gemm<MODE_GATE_UP>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem))) return e;
  if ((e = cudaFuncSetAttribute(pf_gemm<MODE_DOWN>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem))) return e;
  pf_prep<<<t, 256, 0, st>>>(p);
  pf_gemm<MODE_ROUTER><<<((p.E + 127) / 128) * ((t + 127) / 128), PT, kSmem, st>>>(p);
  pf_topk<<<(t + 7) / 8, 256, 0, st>>>(p);
  pf_group<<<1, 1024, 0, st>>>(p);
  pf_fill<<<nch, 32, (size_t)p.E * 4, st>>>(p);
  if (!p.route_only) {
    if ((e = cudaMemsetAsync(p.Y, 0, (size_t)t * p.H * 4, st))) return e;
    pf_gemm<MODE_GATE_UP><<<items * (p.I / 64), PT, kSmem, st>>>(p);
    pf_gemm<MODE_DOWN><<<items * (p.H / 128), PT, kSmem, st>>>(p);
    pf_final<<<1024, 256, 0, st>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace moe
