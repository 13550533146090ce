// decode.cu -- persistent decode / speculative-verify kernel for nb <= 4 rows.
//
// One cooperative grid (one CTA per SM) runs every layer of a call.  Per layer:
//   R  each CTA loads the layer input (applying the unit RMSNorm when asked),
//      stages it as bf16 hi/lo tensor-core fragments, and computes its share of
//      the router rows (bf16 router x fp32 input on CUDA cores) plus the
//      shared-gate dot; a release counter publishes the logits.
//   T  every CTA waits for all router rows, then computes top-k, softmax and
//      the union itself (identical in every CTA, so no second grid-wide
//      handshake); CTA 0 publishes slot table, weight map and ids.
//   G  gate_up units (internal slot, 16 gate rows + the matching 16 up rows)
//   D  down units (slot, 64 output rows).
// Weight tiles of the units reach shared memory through bulk (TMA) copies:
// one thread keeps a ring of `stages` units in flight, so HBM streams while
// the warps compute.  The shared expert's first gate_up units do not depend
// on routing and are requested before the layer input is even available.
// Codes are expanded to exact bf16 integers and multiplied on the tensor
// cores against the staged activations; scale and bias apply per 64-code
// group in fp32; h = silu(gate) * up is stored as bf16 hi/lo fragments for
// the down projection; the down result is scaled by the routing weight (or
// the shared gate) and kept per slot; the last unit of each 64-row range
// (atomic ticket) sums the slots in a fixed order, adds the residual and
// writes the layer output.  No float atomics: results are reproducible.
// Every wait has a deadline (%globaltimer); on expiry the kernel records
// MOE_ETIMEOUT and returns instead of hanging.
//
// Sources: `Gpu::router_b`, `Gpu::experts_b`, `encode_block`, the `slot_tab`
// / `wmap` fields (struct Gpu page), `union_of`, `struct Q`, `MAX_NB`,
// `SLOT_STRIDE` (gpu.rs source page).
#include <cuda_runtime.h>

#include "codec.cuh"
#include "decode.cuh"

namespace moe {
namespace {

constexpr int NT = 512;
constexpr int NW = NT / 32;
constexpr int MAXIT = 4;
constexpr int kTscWords = 2 * 16 * 33 > 2 * 8 * 65 ? 2 * 16 * 33 : 2 * 8 * 65;  // transposed scales of a unit
constexpr int kProducerWarp = 1;  // issues the bulk copies (thread 0 does the cross-CTA releases)

// Shared-memory row pitch of a staged code row of rb bytes: padded so that
// the lanes of one load phase (two rows x 64 B at 4 bits, four rows x 32 B
// at 2 bits, eight rows x 4 x 4 B at 12-byte stride at 3 bits) hit distinct
// banks: pitch = 64, 32, 16 (mod 128) for 4, 2, 3 bits.
__host__ __device__ constexpr int code_pitch(int rb, int bits) {
  const int target = bits == 4 ? 64 : (bits == 2 ? 32 : 16);
  return rb + ((target - rb % 128) + 128) % 128;
}
constexpr unsigned FULL = 0xffffffffu;
constexpr uint32_t kResidual = 1, kPrenorm = 2;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}

__device__ __forceinline__ uint32_t orderable(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// bf16 hi / lo split of an fp32 value: v ~= hi + lo to 16 significant bits.
__device__ __forceinline__ uint32_t split_part(float v, int hl) {
  uint32_t h = f2bf(v);
  return hl ? f2bf(v - __uint_as_float(h << 16)) : h;
}

// (a, b) -> bf16x2 hi = (bf16(a), bf16(b)) and lo = bf16 of the remainders (a first, low half)
__device__ __forceinline__ void split2(float a, float b, uint32_t &hi, uint32_t &lo) {
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(hi) : "f"(b), "f"(a));
  const float ra = a - __uint_as_float(hi << 16), rb = b - __uint_as_float(hi & 0xffff0000u);
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(lo) : "f"(rb), "f"(ra));
}

// ceil(c*n/g), floor(c*n/g); c*n stays far below 2^31 for every shape accepted
__device__ __forceinline__ int cdiv_mul(int c, int n, int g) { return (c * n + g - 1) / g; }
__device__ __forceinline__ int fdiv_mul(int c, int n, int g) { return c * n / g; }

// Thread 0: poll *p until it reaches target, the call aborts, or the deadline passes.
__device__ bool wait_geq(const unsigned *p, unsigned target, const FwdParams &P) {
  const uint64_t t0 = globaltimer();
  unsigned spins = 0;
  while (ld_acquire(p) < target) {
    if ((++spins & 31u) == 0) {
      if (ld_volatile_int(P.status) != 0) return false;
      if (globaltimer() - t0 > P.timeout_ns) {
        atomicCAS(P.status, 0, kStatusTimeout);
        return false;
      }
    }
  }
  return true;
}

__device__ bool cta_wait(const unsigned *p, unsigned target, const FwdParams &P, volatile int *flag) {
  if (threadIdx.x == 0) *flag = wait_geq(p, target, P);
  __syncthreads();
  const bool ok = *flag;
  __syncthreads();
  return ok;
}

// All threads: publish this CTA's writes, then add v to *p (release).
__device__ void cta_signal(unsigned *p, unsigned v) {
  __syncthreads();
  if (threadIdx.x == 0) red_release_add(p, v);
}

// All threads: wait for ring stage `u` (its copies landed).  A wait that
// passes the deadline records MOE_ETIMEOUT and keeps waiting (the copies
// in flight target this CTA's shared memory) for up to one more deadline.
__device__ bool stage_wait(uint64_t *bar, uint32_t parity, const FwdParams &P) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  bool late = false;
  while (!mbar_try_wait(bar, parity)) {
    const uint64_t dt = globaltimer() - t0;
    if (!late && dt > P.timeout_ns) {
      atomicCAS(P.status, 0, kStatusTimeout);
      late = true;
    }
    if (dt > 2 * P.timeout_ns) return false;
  }
  return !late;
}

// Thread 0, on an error return: wait (bounded) for the copies still in
// flight into this CTA's ring, units [from, to) of the call's sequence.
__device__ void drain_ring(uint64_t *bars, unsigned from, unsigned to, int S, const FwdParams &P) {
  if (threadIdx.x != 0) return;  // any one thread keeps the CTA (and its ring) alive until the copies land
  for (unsigned u = from; u < to; u++) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(&bars[u % S], (u / S) & 1u))
      if (globaltimer() - t0 > P.timeout_ns) return;
  }
}

// ------------------------------------------------------------ activation staging

// Thread (blk, b, t) turns the 32 inputs x[b][blk*128 + 32t .. +32) into the
// bf16 hi / lo A-fragment registers of lanes (hl*4 + b, t) for the 8 MMA
// steps of the block, in codec B's pair order, each input pre-scaled by the
// 2^-s of its pair half (exact).  Also per 64-input group: xs = sum of x
// (bias term) and cs = 128 * sum of 2^-s x (the offset the codes carry).
template <int B>
__device__ void stage_frags(const float *xf, int H, int nb, uint2 *xa, float *xs, float *cs) {
  const int nblk = H / 128;
  for (int j = threadIdx.x; j < nblk * 16; j += NT) {
    const int t = j & 3, b = (j >> 2) & 3, blk = j >> 4;
    float v[32];
    if (b < nb) {
      const float4 *src = reinterpret_cast<const float4 *>(xf + b * H + blk * 128 + 32 * t);
#pragma unroll
      for (int i = 0; i < 8; i++) {
        const float4 q = src[i];
        v[4 * i] = q.x, v[4 * i + 1] = q.y, v[4 * i + 2] = q.z, v[4 * i + 3] = q.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; i++) v[i] = 0.f;
    }
    float sx = 0.f, sc = 0.f;
#pragma unroll
    for (int i = 0; i < 32; i++) sx += v[i];
#pragma unroll
    for (int m = 0; m < 8; m++) {
      const int p0 = 2 * m, p1 = 2 * m + 1;
      const float a0 = v[Codec<B>::lo(p0)] * pow2neg(Codec<B>::slo(p0));
      const float a1 = v[Codec<B>::hi(p0)] * pow2neg(Codec<B>::shi(p0));
      const float a2 = v[Codec<B>::lo(p1)] * pow2neg(Codec<B>::slo(p1));
      const float a3 = v[Codec<B>::hi(p1)] * pow2neg(Codec<B>::shi(p1));
      sc += (a0 + a1) + (a2 + a3);
      uint32_t hi0, lo0, hi1, lo1;
      split2(a0, a1, hi0, lo0);
      split2(a2, a3, hi1, lo1);
      xa[(blk * 8 + m) * 32 + 4 * b + t] = make_uint2(hi0, hi1);
      xa[(blk * 8 + m) * 32 + 4 * (4 + b) + t] = make_uint2(lo0, lo1);
    }
    sx += __shfl_xor_sync(FULL, sx, 1);
    sc += __shfl_xor_sync(FULL, sc, 1);
    if ((t & 1) == 0) {
      if (xs) xs[b * (H / 64) + 2 * blk + (t >> 1)] = sx;
      cs[b * (H / 64) + 2 * blk + (t >> 1)] = 128.f * sc;
    }
  }
}

// ------------------------------------------------------------ tensor-core items

// The four A registers of each MMA step: lanes with t < 2 carry codes of the
// block's first group (A rows 0..7), lanes with t >= 2 of its second group
// (rows 8..15); the other half of each lane's A fragment is zero.
struct AFrag {
  uint32_t r[8][4];
};
__device__ __forceinline__ void make_afrag(const uint2 (&x)[8], bool lowT, AFrag &A) {
#pragma unroll
  for (int m = 0; m < 8; m++) {
    A.r[m][0] = lowT ? x[m].x : 0u;
    A.r[m][1] = lowT ? 0u : x[m].x;
    A.r[m][2] = lowT ? x[m].y : 0u;
    A.r[m][3] = lowT ? 0u : x[m].y;
  }
}

// One item: 8 weight rows x one block of 128 inputs.  Codes and the scale /
// bias pairs come from the stage in shared memory; A holds the activation
// fragments of the block.  Returns, in lanes 0..15 (b = lane/4), the results
// of rows 2t and 2t+1 of the item (already summed over hi and lo parts).
// ci0 / ci1: accumulator start of the lane's rows for the block's two groups
// (minus the offset sum on hi lanes, 0 on lo lanes); xs0 / xs1: the groups'
// input sums on hi lanes, 0 on lo lanes (so the bias enters once).
template <int B>
__device__ __forceinline__ void item_compute(const uint8_t *codes_row, const uint32_t *sc, const uint32_t *bi,
                                             const AFrag &A, float ci0, float ci1, float xs0,
                                             float xs1, float &o0, float &o1) {
  uint32_t w[Codec<B>::kWords];
  if constexpr (B == 4) {
    const uint4 v = *reinterpret_cast<const uint4 *>(codes_row);
    w[0] = v.x, w[1] = v.y, w[2] = v.z, w[3] = v.w;
  } else if constexpr (B == 2) {
    const uint2 v = *reinterpret_cast<const uint2 *>(codes_row);
    w[0] = v.x, w[1] = v.y;
  } else {
    const uint32_t *p = reinterpret_cast<const uint32_t *>(codes_row);
    w[0] = p[0], w[1] = p[1], w[2] = p[2];
  }
  const uint32_t s0 = sc[0], s1 = sc[1], b0 = bi[0], b1 = bi[1];
  uint32_t bf[16];
  Codec<B>::unpack(w, bf);
  float d[4] = {ci0, ci0, ci1, ci1}, e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int m = 0; m < 8; m += 2) {
    mma_bf16_16816(d, A.r[m][0], A.r[m][1], A.r[m][2], A.r[m][3], bf[2 * m], bf[2 * m + 1]);
    mma_bf16_16816(e, A.r[m + 1][0], A.r[m + 1][1], A.r[m + 1][2], A.r[m + 1][3], bf[2 * m + 2], bf[2 * m + 3]);
  }
#pragma unroll
  for (int i = 0; i < 4; i++) d[i] += e[i];
  float r0 = bf16lo(s0) * d[0] + bf16hi(s0) * d[2];
  float r1 = bf16lo(s1) * d[1] + bf16hi(s1) * d[3];
  r0 += bf16lo(b0) * xs0 + bf16hi(b0) * xs1;
  r1 += bf16lo(b1) * xs0 + bf16hi(b1) * xs1;
  o0 = r0 + __shfl_xor_sync(FULL, r0, 16);
  o1 = r1 + __shfl_xor_sync(FULL, r1, 16);
}

// items per warp: the smallest power of two covering all items, capped at ntiles
__device__ __forceinline__ int items_per_warp(int nitems, int ntiles) {
  const int need = (nitems + NW - 1) / NW;
  int ipw = 1;
  while (ipw < need) ipw *= 2;
  return ipw < ntiles ? ipw : ntiles;
}

// Stage layout of a gate_up unit: codes of 16 gate rows then 16 up rows
// (32 rows), then their scales (32 rows), then their biases (32 rows).
// Writes red[(kb*4 + nt)*32 + row*4 + b].
#ifdef MOE_DEBUG_CYCLES
__device__ long long g_dbg_cycles[64];
#define MOE_DBG(k) if (blockIdx.x == 0 && (threadIdx.x & 31) == 0 && (threadIdx.x >> 5) < 4) g_dbg_cycles[(threadIdx.x >> 5) * 16 + (k)] = clock64();
#else
#define MOE_DBG(k)
#endif

template <int B>
__device__ void gate_up_compute(const uint8_t *st, const uint32_t *T, int H, const uint2 *xa, const float *xs,
                                const float *cs, int nb, float *red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3, b = g & 3;
  const int nblk = H / 128;
  const int nitems = nblk * 4;
  const int ipw = items_per_warp(nitems, 4);
  const int i0 = warp * ipw;
  if (i0 >= nitems) return;
  const int kb = i0 >> 2;
  const int pitch = code_pitch(H * B / 8, B), np = H / 128;
  MOE_DBG(0)
  uint2 a[8];
#pragma unroll
  for (int m = 0; m < 8; m++) a[m] = xa[(kb * 8 + m) * 32 + lane];
  AFrag A;
  make_afrag(a, t < 2, A);
  MOE_DBG(1)
  const bool hl0 = g < 4;
  const float xs0 = hl0 ? xs[b * (H / 64) + 2 * kb] : 0.f, xs1 = hl0 ? xs[b * (H / 64) + 2 * kb + 1] : 0.f;
  const float ci0 = hl0 ? -cs[b * (H / 64) + 2 * kb] : 0.f, ci1 = hl0 ? -cs[b * (H / 64) + 2 * kb + 1] : 0.f;
  const uint32_t *sc = T + kb * 33, *bi = T + (np + kb) * 33;
#pragma unroll 1
  for (int k = 0; k < ipw; k++) {
    {
      const int nt = (i0 & 3) + k;
      float o0, o1;
      item_compute<B>(st + (8 * nt + g) * pitch + kb * (16 * B) + t * (4 * B), sc + 8 * nt + 2 * t,
                      bi + 8 * nt + 2 * t, A, ci0, ci1, xs0, xs1, o0, o1);
      if (lane < 16 && b < nb) {
        red[(kb * 4 + nt) * 32 + (2 * t) * 4 + b] = o0;
        red[(kb * 4 + nt) * 32 + (2 * t + 1) * 4 + b] = o1;
      }
      MOE_DBG(2 + k)
    }
  }
}

// Stage layout of a down unit: codes of 64 output rows, their scales, their
// biases.  a[] / hs0 / hs1: this warp's h fragments and group sums.
template <int B>
__device__ void down_compute(const uint8_t *st, const uint32_t *T, int I, const uint2 (&x)[8], float ci0, float ci1,
                             float hs0, float hs1, int nb, float *red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3, b = g & 3;
  const int nitems = (I / 128) * 8;
  const int ipw = items_per_warp(nitems, 8);
  const int i0 = warp * ipw;
  if (i0 >= nitems) return;
  const int kb = i0 >> 3;
  const int pitch = code_pitch(I * B / 8, B), np = I / 128;
  AFrag A;
  make_afrag(x, t < 2, A);
  const uint32_t *sc = T + kb * 65, *bi = T + (np + kb) * 65;
#pragma unroll 1
  for (int k = 0; k < ipw; k++) {
    {
      const int nt = (i0 & 7) + k;
      float o0, o1;
      item_compute<B>(st + (8 * nt + g) * pitch + kb * (16 * B) + t * (4 * B), sc + 8 * nt + 2 * t,
                      bi + 8 * nt + 2 * t, A, ci0, ci1, hs0, hs1, o0, o1);
      if (lane < 16 && b < nb) {
        red[(kb * 8 + nt) * 32 + (2 * t) * 4 + b] = o0;
        red[(kb * 8 + nt) * 32 + (2 * t + 1) * 4 + b] = o1;
      }
    }
  }
}

// ------------------------------------------------------------ routing

// Top-k of one row of E <= 1024 logits (ties to the lower id), then softmax
// over the k chosen.  Lane l holds ids [l*P, l*P+P) as order-preserving keys
// in registers; each round one warp max picks the winner, whose lane alone
// rescans its keys.
template <int PM>
__device__ void topk_warp(const float *lg, int E, int K, int *idx, float *w) {
  const int lane = threadIdx.x & 31;
  const int P = (E + 31) / 32;
  uint32_t key[PM];
#pragma unroll
  for (int i = 0; i < PM; i++) {
    const int e = lane * P + i;
    key[i] = (i < P && e < E) ? orderable(lg[e]) : 0u;
  }
  uint32_t bk = 0;
  int bi = 0;
#pragma unroll
  for (int i = 0; i < PM; i++)
    if (key[i] > bk) bk = key[i], bi = i;
#pragma unroll 1
  for (int r = 0; r < K; r++) {
    const uint32_t m = __reduce_max_sync(FULL, bk);
    const int wl = __ffs(__ballot_sync(FULL, bk == m)) - 1;
    if (lane == wl) {
      idx[r] = lane * P + bi;
      w[r] = lg[lane * P + bi];
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
  __syncwarp();
  const float mx = w[0];
  const float ev = lane < K ? expf(w[lane] - mx) : 0.f;
  const float z = warp_sum(ev);
  __syncwarp();
  if (lane < K) w[lane] = ev / z;
  __syncwarp();
}

// Union of the [nb][K] ids in first-seen order (warp 0).  Writes uni[],
// wm[b][slot] and *nu = U.  rk is 64 ints of scratch.  Position p = b*K + r.
__device__ void union_warp(const int *sidx, const float *sw, int nb, int K, int *uni, float *wm, int *rk,
                           volatile int *nu) {
  const int lane = threadIdx.x & 31;
  for (int j = lane; j < 256; j += 32) wm[j] = 0.f;
  int id[2], first[2], fpos[2], pb[2], pr[2];
#pragma unroll
  for (int h = 0; h < 2; h++) {
    const int pos = lane + 32 * h;
    int b = 0, r = pos;
    while (b < nb && r >= K) r -= K, b++;
    pb[h] = b, pr[h] = r;
    id[h] = -1, first[h] = 0, fpos[h] = pos;
    if (b < nb) {
      id[h] = sidx[b * 32 + r];
      first[h] = 1;
      int q = 0;
      for (int b2 = 0; b2 <= b && first[h]; b2++) {
        const int rend = b2 < b ? K : r;
        for (int r2 = 0; r2 < rend; r2++, q++) {
          if (sidx[b2 * 32 + r2] == id[h]) {
            first[h] = 0;
            fpos[h] = q;
            break;
          }
        }
      }
    }
  }
  const uint32_t b0 = __ballot_sync(FULL, first[0]), b1 = __ballot_sync(FULL, first[1]);
  const uint32_t lt = (1u << lane) - 1u;
  if (first[0]) rk[lane] = __popc(b0 & lt);
  if (first[1]) rk[lane + 32] = __popc(b0) + __popc(b1 & lt);
  __syncwarp();
#pragma unroll
  for (int h = 0; h < 2; h++) {
    if (pb[h] < nb) {
      const int slot = rk[fpos[h]];
      if (first[h]) uni[slot] = id[h];
      wm[pb[h] * 64 + slot] = sw[pb[h] * 32 + pr[h]];
    }
  }
  if (lane == 0) *nu = __popc(b0) + __popc(b1);
  __syncwarp();
}

// ------------------------------------------------------------ unit schedule

struct Sched {
  int hsi, ups, nrt, U, nslots;
  int early;        // shared gate_up units assigned before routing
  int nA, sA0;      // early shared units of this CTA
  int nB, rB0;      // gate_up units after routing (routed only if early, else shared + routed)
  int nD, d0;       // down units
  __device__ int n() const { return nA + nB + nD; }
};

struct UnitDesc {
  int down, slot, row0;  // row0: gate_up chunk start (inter rows) or down output row start
  const uint8_t *rec;
  QOff q;
  int bits;
};

template <int BITS>
__device__ __forceinline__ UnitDesc get_unit(int q, const Sched &s, const LayerP &L,
                                             const uint8_t *const *rect) {
  UnitDesc d;
  if (q < s.nA) {
    d.down = 0, d.slot = 0, d.row0 = (s.sA0 + q) * 16;
  } else if (q < s.nA + s.nB) {
    const int r = s.rB0 + (q - s.nA);
    d.down = 0;
    d.slot = (s.early ? s.hsi : 0) + r / s.ups;
    d.row0 = (r % s.ups) * 16;
  } else {
    const int r = s.d0 + (q - s.nA - s.nB);
    d.down = 1, d.slot = r / s.nrt, d.row0 = (r % s.nrt) * 64;
  }
  const bool shared = s.hsi && d.slot == 0;
  d.rec = shared ? L.srec : rect[d.slot];
  d.q = shared ? (d.down ? L.sdn : L.sgu) : (d.down ? L.dn : L.gu);
  d.bits = shared ? 4 : BITS;
  return d;
}

// Producer warp: request the weight tile of one unit into its ring stage.
// Code rows land at the padded pitch (one bulk copy per row, the warp's
// lanes issuing in parallel); scales and biases land row-major.
__device__ void issue_unit(const UnitDesc &d, int H, int I, uint8_t *st, uint64_t *bar, int *status) {
  const int lane = threadIdx.x & 31;
  if (d.rec == nullptr || ((uintptr_t)d.rec & 15u)) {
    if (lane == 0) {
      atomicCAS(status, 0, kStatusDevice);
      mbar_expect_tx(bar, 0);  // completes the phase with no bytes
    }
    return;
  }
  const int inp = d.down ? I : H;
  const uint32_t rb = inp * d.bits / 8, sp = inp / 32, pitch = code_pitch(rb, d.bits);
  const int rows = d.down ? 64 : 32;
  if (lane == 0) mbar_expect_tx(bar, rows * (rb + 2 * sp));
  __syncwarp();
  const uint8_t *c = d.rec + d.q.w;
  for (int r = lane; r < rows; r += 32) {
    // gate_up: rows 0..15 the gate rows row0.., 16..31 the up rows I+row0..
    const int src = d.down ? d.row0 + r : (r < 16 ? d.row0 + r : I + d.row0 + r - 16);
    bulk_g2s(st + r * pitch, c + (size_t)src * rb, rb, bar);
  }
  if (lane == 0) {
    uint8_t *sdst = st + rows * pitch;
    if (d.down) {
      bulk_g2s(sdst, d.rec + d.q.s + (size_t)d.row0 * sp, 64 * sp, bar);
      bulk_g2s(sdst + 64 * sp, d.rec + d.q.b + (size_t)d.row0 * sp, 64 * sp, bar);
    } else {
      bulk_g2s(sdst, d.rec + d.q.s + (size_t)d.row0 * sp, 16 * sp, bar);
      bulk_g2s(sdst + 16 * sp, d.rec + d.q.s + (size_t)(I + d.row0) * sp, 16 * sp, bar);
      bulk_g2s(sdst + 32 * sp, d.rec + d.q.b + (size_t)d.row0 * sp, 16 * sp, bar);
      bulk_g2s(sdst + 48 * sp, d.rec + d.q.b + (size_t)(I + d.row0) * sp, 16 * sp, bar);
    }
  }
}

// All threads: transpose the unit's scales and biases, [row][pair] u32
// (two groups of a block per u32) -> T[which][pair][row] with row stride
// rows + 1, so that an item's lanes read their rows without conflicts.
__device__ void transpose_scales(const uint8_t *sd, int rows, int npair, uint32_t *T) {
  const uint32_t *src = reinterpret_cast<const uint32_t *>(sd);
  const int per = rows * npair;
  for (int e = threadIdx.x; e < 2 * per; e += NT) {
    const int which = e / per, rem = e - which * per;
    const int r = rem / npair, kb = rem - r * npair;
    T[(which * npair + kb) * (rows + 1) + r] = src[e];
  }
}

// ------------------------------------------------------------ the kernel

template <int BITS>
__global__ void __launch_bounds__(NT, 1) decode_kernel(const __grid_constant__ FwdParams P) {
  extern __shared__ __align__(128) unsigned char sm[];
  const int H = P.H, E = P.E, K = P.K, I = P.I, nb = P.nb;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  const int nblkH = H / 128, nblkI = I / 128;
  const int E1 = (E + 1 + 3) & ~3;
  const int ng = H / 64;
  const int S = P.stages;

  uint8_t *stages = sm;                                                  // [S][stage_bytes]
  float *xf = reinterpret_cast<float *>(sm + (size_t)S * P.stage_bytes);  // [4][H]
  uint2 *xa = reinterpret_cast<uint2 *>(xf + 4 * H);                     // [nblkH][8][32] routed codec order
  uint2 *xa4 = BITS == 4 ? xa : xa + nblkH * 256;                        // shared (4-bit) order
  float *xs = reinterpret_cast<float *>(xa4 + nblkH * 256);              // [4][H/64] group sums of x
  float *cs = xs + 4 * ng;                                               // [4][H/64] offset sums, routed order
  float *cs4 = cs + 4 * ng;                                              // [4][H/64] offset sums, 4-bit order
  float *lg = cs4 + 4 * ng;                                              // [4][E1]
  float *red = lg + 4 * E1;                                              // [2048]
  int *sidx = reinterpret_cast<int *>(red + 2048);                       // [4][32]
  float *sw = reinterpret_cast<float *>(sidx + 128);                     // [4][32]
  int *uni = reinterpret_cast<int *>(sw + 128);                          // [64]
  float *wm = reinterpret_cast<float *>(uni + 64);                       // [4][64]
  float *gam = wm + 256;                                                 // [4]
  volatile int *sflag = reinterpret_cast<volatile int *>(gam + 4);       // [12]
  uint64_t *bars = reinterpret_cast<uint64_t *>(gam + 16);               // [kMaxStages]
  const uint8_t **rect = reinterpret_cast<const uint8_t **>(bars + kMaxStages);  // [64] slot -> record
  uint32_t *tsc = reinterpret_cast<uint32_t *>(rect + 64);                      // [1056] transposed scales
  uint64_t *eaddr_s = reinterpret_cast<uint64_t *>(tsc + kTscWords);           // [E] expert addresses

  if (tid == 0) {
    for (int s = 0; s < S; s++) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  __syncthreads();

  unsigned qbase = 0;  // units requested so far in this call (ring position)
  for (int l = 0; l < P.nl; l++) {
#define MOE_STAMP(k)                                                                             \
  if (P.trace && tid == 0 && cta < kTraceCtas)                                                   \
    P.trace[((size_t)l * kTraceCtas + cta) * kTracePhases + (k)] = globaltimer();
    MOE_STAMP(0)
    const LayerP &L = P.L[l];
    unsigned *cnt = P.cnt + (size_t)l * kCntPerLayer;
    const bool hs = L.sgate != nullptr;
    const float *src = l == 0 ? P.x : P.xbuf + (size_t)l * 4 * H;
    float *dst = l == P.nl - 1 ? P.out : P.xbuf + (size_t)(l + 1) * 4 * H;

    Sched s;
    s.hsi = hs ? 1 : 0;
    s.ups = I / 16;
    s.nrt = H / 64;
    s.early = hs && !P.route_only && (K + 1) * s.ups >= G;
    s.sA0 = s.early ? cdiv_mul(cta, s.ups, G) : 0;
    s.nA = s.early ? cdiv_mul(cta + 1, s.ups, G) - s.sA0 : 0;
    s.nB = s.nD = s.rB0 = s.d0 = 0;
    s.U = 0;
    int issued = 0;
    if (warp == kProducerWarp) {
      for (; issued < s.nA && issued < S; issued++) {
        const unsigned u = qbase + issued;
        issue_unit(get_unit<BITS>(issued, s, L, rect), H, I, stages + (size_t)(u % S) * P.stage_bytes,
                   &bars[u % S], P.status);
      }
    }
    issued = s.nA < S ? s.nA : S;

    // ---- R: input, norm, fragments, router rows
    if (l > 0 && !cta_wait(P.cnt + (size_t)(l - 1) * kCntPerLayer + kCntRows, (unsigned)(H / 64), P, sflag)) {
      drain_ring(bars, qbase, qbase + issued, S, P);
      return;
    }
    MOE_STAMP(1)
    {
      // one round trip: each thread loads up to 4 float4 of the nb rows
      const int n4 = nb * H / 4, h4 = H / 4;
      const float4 *src4 = reinterpret_cast<const float4 *>(src);
      float4 v[4];
#pragma unroll
      for (int k = 0; k < 4; k++) {
        const int i = tid + k * NT;
        v[k] = i < n4 ? __ldcg(src4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      if (L.flags & kPrenorm) {
        // per-row sums of squares: thread partials -> warp sums -> CTA sums (fixed order)
        float ss[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < 4; k++) {
          const int i = tid + k * NT;
          if (i < n4) {
            const float q = v[k].x * v[k].x + v[k].y * v[k].y + v[k].z * v[k].z + v[k].w * v[k].w;
            ss[i / h4] += q;
          }
        }
#pragma unroll
        for (int b = 0; b < 4; b++) ss[b] = warp_sum(ss[b]);
        if (lane == 0)
          for (int b = 0; b < 4; b++) red[warp * 4 + b] = ss[b];
        __syncthreads();
        if (tid < 4) {
          float t = 0.f;
          for (int w = 0; w < NW; w++) t += red[w * 4 + tid];
          red[64 + tid] = 1.0f / sqrtf(t / (float)H + 1e-6f);
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < 4; k++) {
          const int i = tid + k * NT;
          if (i < n4) {
            const float r = red[64 + i / h4];
            v[k].x *= r, v[k].y *= r, v[k].z *= r, v[k].w *= r;
          }
        }
      }
      float4 *xf4 = reinterpret_cast<float4 *>(xf);
#pragma unroll
      for (int k = 0; k < 4; k++) {
        const int i = tid + k * NT;
        if (i < H) xf4[i] = v[k];  // rows b >= nb hold zeros
      }
    }
    __syncthreads();
    stage_frags<BITS>(xf, H, nb, xa, xs, cs);
    if (BITS != 4 && hs) stage_frags<4>(xf, H, nb, xa4, nullptr, cs4);
    const int R = E + s.hsi;
    const int rr0 = fdiv_mul(cta, R, G), rr1 = fdiv_mul(cta + 1, R, G);
    const int nch = H / 256;
    const int nitem = (rr1 - rr0) * nch;
    __syncthreads();
    MOE_STAMP(2)
    {
      // every router load of this warp in flight at once (<= 4 items per warp)
      uint4 wv[4];
#pragma unroll
      for (int k = 0; k < 4; k++) {
        const int it = warp + k * NW;
        if (it < nitem) {
          const int row = rr0 + it / nch, ch = it % nch;
          const uint16_t *wrow = row < E ? L.router + (size_t)row * H : L.sgate;
          wv[k] = ldg_stream4(wrow + ch * 256 + lane * 8);
        }
      }
#pragma unroll
      for (int k = 0; k < 4; k++) {
        const int it = warp + k * NW;
        if (it < nitem) {
          const int ch = it % nch;
          const float wf[8] = {bf16lo(wv[k].x), bf16hi(wv[k].x), bf16lo(wv[k].y), bf16hi(wv[k].y),
                               bf16lo(wv[k].z), bf16hi(wv[k].z), bf16lo(wv[k].w), bf16hi(wv[k].w)};
          for (int b = 0; b < nb; b++) {
            const float4 *xp = reinterpret_cast<const float4 *>(xf + b * H + ch * 256 + lane * 8);
            const float4 x0 = xp[0], x1 = xp[1];
            float acc = wf[0] * x0.x + wf[1] * x0.y + wf[2] * x0.z + wf[3] * x0.w + wf[4] * x1.x +
                        wf[5] * x1.y + wf[6] * x1.z + wf[7] * x1.w;
            acc = warp_sum(acc);
            if (lane == 0) red[it * 4 + b] = acc;
          }
        }
      }
    }
    __syncthreads();
    for (int j = tid; j < (rr1 - rr0) * nb; j += NT) {
      const int r = j / nb, b = j % nb;
      float sum = 0.f;
      for (int ch = 0; ch < nch; ch++) sum += red[(r * nch + ch) * 4 + b];
      P.logits[((size_t)l * 4 + b) * (E + 1) + rr0 + r] = sum;
    }
    if (rr1 > rr0) cta_signal(cnt + kCntRouter, (unsigned)(rr1 - rr0));
    MOE_STAMP(3)
    // expert addresses (for the slot table) while the other CTAs finish their router rows
    for (int e = tid; e < E; e += NT) eaddr_s[e] = L.eaddr[e];

    // ---- T: top-k, softmax, union
    if (!cta_wait(cnt + kCntRouter, (unsigned)(R + (P.withhold ? 1 : 0)), P, sflag)) {
      drain_ring(bars, qbase, qbase + issued, S, P);
      return;
    }
    MOE_STAMP(4)
    for (int i = tid; i < nb * (E + 1); i += NT) {
      const int b = i / (E + 1), e = i % (E + 1);
      lg[b * E1 + e] = e < R ? __ldcg(P.logits + ((size_t)l * 4 + b) * (E + 1) + e) : 0.f;
    }
    __syncthreads();
    MOE_STAMP(8)
    if (warp < nb) {
      if (E <= 128)
        topk_warp<4>(lg + warp * E1, E, K, sidx + warp * 32, sw + warp * 32);
      else if (E <= 256)
        topk_warp<8>(lg + warp * E1, E, K, sidx + warp * 32, sw + warp * 32);
      else if (E <= 512)
        topk_warp<16>(lg + warp * E1, E, K, sidx + warp * 32, sw + warp * 32);
      else
        topk_warp<32>(lg + warp * E1, E, K, sidx + warp * 32, sw + warp * 32);
    }
    if (tid < 4) gam[tid] = (hs && tid < nb) ? 1.f / (1.f + expf(-lg[tid * E1 + E])) : 0.f;
    __syncthreads();
    MOE_STAMP(9)
    if (warp == 0) union_warp(sidx, sw, nb, K, uni, wm, reinterpret_cast<int *>(red), sflag + 1);
    __syncthreads();
    MOE_STAMP(10)
    s.U = sflag[1];
    if (tid < s.U) rect[tid + s.hsi] = reinterpret_cast<const uint8_t *>(eaddr_s[uni[tid]]);
    if (cta == 0) {
      if (P.slot_tab)
        for (int j = tid; j < kSlotStride; j += NT) {
          uint64_t v = j < s.U ? eaddr_s[uni[j]] : 0ull;
          if (j == kSlotStride - 2 || j == kSlotStride - 1) v = (uint64_t)s.U;
          P.slot_tab[(size_t)l * kSlotStride + j] = v;
        }
      if (P.wmap)
        for (int j = tid; j < kMaxNb * kSlotStride; j += NT) P.wmap[(size_t)l * kMaxNb * kSlotStride + j] = wm[j];
      if (P.topk_idx)
        for (int j = tid; j < nb * K; j += NT)
          P.topk_idx[(size_t)l * nb * K + j] = (uint32_t)sidx[(j / K) * 32 + j % K];
      if (P.topk_w)
        for (int j = tid; j < nb * K; j += NT) P.topk_w[(size_t)l * nb * K + j] = sw[(j / K) * 32 + j % K];
      if (P.logits_out)
        for (int j = tid; j < nb * E; j += NT) P.logits_out[j] = lg[(j / E) * E1 + j % E];
    }
    if (P.route_only) continue;

    // ---- schedule of this CTA's units for the layer
    __syncthreads();
    s.nslots = s.U + s.hsi;
    if (s.early) {
      const int T = (s.U + 1) * s.ups;  // shared + routed gate_up units
      s.rB0 = fdiv_mul(cta, T, G) - cdiv_mul(cta, s.ups, G);
      s.nB = fdiv_mul(cta + 1, T, G) - cdiv_mul(cta + 1, s.ups, G) - s.rB0;
    } else {
      const int T = s.nslots * s.ups;
      s.rB0 = fdiv_mul(cta, T, G);
      s.nB = fdiv_mul(cta + 1, T, G) - s.rB0;
    }
    const int ND = s.nslots * s.nrt;
    s.d0 = fdiv_mul(cta, ND, G);
    s.nD = fdiv_mul(cta + 1, ND, G) - s.d0;
    const int n = s.n();
    if (warp == kProducerWarp) {
      for (int q = issued; q < n && q < S; q++) {
        const unsigned u = qbase + q;
        issue_unit(get_unit<BITS>(q, s, L, rect), H, I, stages + (size_t)(u % S) * P.stage_bytes, &bars[u % S],
                   P.status);
      }
    }
    issued = n < S ? n : S;

    // ---- G + D: the unit loop
    MOE_STAMP(5)
    int cur = -1;
    uint2 da[8];
    float hs0 = 0.f, hs1 = 0.f, dc0 = 0.f, dc1 = 0.f;
    for (int q = 0; q < n; q++) {
      if (q == s.nA + s.nB) {
        MOE_STAMP(6)
        if (tid == 0 && l + 1 < P.nl) {
          // the next layer's router rows of this CTA, toward L2 while the down units run
          const LayerP &Ln = P.L[l + 1];
          const int re = rr1 < E ? rr1 : E;
          if (re > rr0) prefetch_l2(Ln.router + (size_t)rr0 * H, (uint32_t)((re - rr0) * H * 2));
          if (rr1 > E && Ln.sgate) prefetch_l2(Ln.sgate, (uint32_t)(H * 2));
        }
      }
      const UnitDesc d = get_unit<BITS>(q, s, L, rect);
      const unsigned u = qbase + q;
      const uint8_t *st = stages + (size_t)(u % S) * P.stage_bytes;
      const bool shared = s.hsi && d.slot == 0;
      if (d.down && d.slot != cur) {
        // h of this slot complete?  then load this warp's fragments of it
        if (!cta_wait(cnt + kCntGu + d.slot, (unsigned)s.ups, P, sflag)) {
          drain_ring(bars, u, qbase + (unsigned)(q + S < n ? q + S : n), S, P);
          return;
        }
        cur = d.slot;
        const int nitems = nblkI * 8;
        const int ipw = items_per_warp(nitems, 8);
        const int kb = (warp * ipw < nitems) ? (warp * ipw) >> 3 : 0;
        const uint2 *hf = reinterpret_cast<const uint2 *>(P.hfrag + (size_t)d.slot * nblkI * 8 * 32 * 4);
#pragma unroll
        for (int m = 0; m < 8; m++) da[m] = __ldcg(hf + (kb * 8 + m) * 32 + lane);
        // sums of the lane's 32 fragment values: as the MMA sees them (scaled
        // by 2^-s: the offset) and unscaled (h itself: the bias term)
        float ssc = 0.f, sun = 0.f;
        if (shared || BITS == 4) {
#pragma unroll
          for (int m = 0; m < 8; m++)
            ssc += bf16lo(da[m].x) + bf16hi(da[m].x) + bf16lo(da[m].y) + bf16hi(da[m].y);
          sun = ssc;
        } else {
#pragma unroll
          for (int m = 0; m < 8; m++) {
            const float v0 = bf16lo(da[m].x), v1 = bf16hi(da[m].x), v2 = bf16lo(da[m].y), v3 = bf16hi(da[m].y);
            ssc += v0 + v1 + v2 + v3;
            sun += v0 * (float)(1 << Codec<BITS>::slo(2 * m)) + v1 * (float)(1 << Codec<BITS>::shi(2 * m)) +
                   v2 * (float)(1 << Codec<BITS>::slo(2 * m + 1)) + v3 * (float)(1 << Codec<BITS>::shi(2 * m + 1));
          }
        }
        // lanes t, t^1 share a group; add the lo part (lane ^ 16)
        ssc += __shfl_xor_sync(FULL, ssc, 1);
        ssc += __shfl_xor_sync(FULL, ssc, 16);
        sun += __shfl_xor_sync(FULL, sun, 1);
        sun += __shfl_xor_sync(FULL, sun, 16);
        const float osc = __shfl_xor_sync(FULL, ssc, 2), oun = __shfl_xor_sync(FULL, sun, 2);
        const bool hl0 = (lane >> 2) < 4, first = (lane & 3) < 2;
        hs0 = hl0 ? (first ? sun : oun) : 0.f;
        hs1 = hl0 ? (first ? oun : sun) : 0.f;
        dc0 = hl0 ? -128.f * (first ? ssc : osc) : 0.f;
        dc1 = hl0 ? -128.f * (first ? osc : ssc) : 0.f;
      }
      if (!__syncthreads_and(stage_wait(&bars[u % S], (u / S) & 1u, P))) {
        drain_ring(bars, u + 1, qbase + (unsigned)(q + S < n ? q + S : n), S, P);
        return;
      }
      if (q == 0) MOE_STAMP(11)
      const bool ok = d.rec != nullptr && ((uintptr_t)d.rec & 15u) == 0;
      if (ok) {
        const int rows = d.down ? 64 : 32, inp = d.down ? I : H;
        transpose_scales(st + rows * code_pitch(inp * d.bits / 8, d.bits), rows, inp / 128, tsc);
      }
      __syncthreads();
      if (ok) {
        if (!d.down) {
          if (shared)
            gate_up_compute<4>(st, tsc, H, xa4, xs, BITS == 4 ? cs : cs4, nb, red);
          else
            gate_up_compute<BITS>(st, tsc, H, xa, xs, cs, nb, red);
        } else {
          if (shared)
            down_compute<4>(st, tsc, I, da, dc0, dc1, hs0, hs1, nb, red);
          else
            down_compute<BITS>(st, tsc, I, da, dc0, dc1, hs0, hs1, nb, red);
        }
      }
      __syncthreads();
      if (q == 0) MOE_STAMP(12)
      // the stage is free: request the unit S places ahead into it
      if (warp == kProducerWarp && q + S < n) {
        issue_unit(get_unit<BITS>(q + S, s, L, rect), H, I, stages + (size_t)(u % S) * P.stage_bytes, &bars[u % S],
                   P.status);
      }
      if (!d.down) {
        // h = silu(gate) * up for 16 rows x nb, scattered as bf16 hi/lo A
        // fragments in the pair order of this slot's down codec
        // lanes (row i of 32 = 16 gate + 16 up, b, kb-part): sums over the blocks
        {
          const int i = tid >> 4, kp = tid & 15;  // 512 threads = 32 rows x 16 parts
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
          for (int kb = kp; kb < nblkH; kb += 16) {
            const float4 r4 = *reinterpret_cast<const float4 *>(&red[(kb * 4 + (i >> 3)) * 32 + (i & 7) * 4]);
            acc[0] += r4.x, acc[1] += r4.y, acc[2] += r4.z, acc[3] += r4.w;
          }
#pragma unroll
          for (int b = 0; b < 4; b++)
#pragma unroll
            for (int o = 8; o; o >>= 1) acc[b] += __shfl_xor_sync(FULL, acc[b], o);
          __syncthreads();
          if (kp == 0) *reinterpret_cast<float4 *>(&red[i * 4]) = make_float4(acc[0], acc[1], acc[2], acc[3]);
          __syncthreads();
        }
        if (tid < 16 * nb) {
          const int i = tid & 15, b = tid >> 4;
          const float gsum = red[i * 4 + b], usum = red[(16 + i) * 4 + b];
          const float h = ok ? gsum / (1.f + expf(-gsum)) * usum : 0.f;
          const int pos = d.row0 + i;
          const int blk = pos >> 7, c = pos & 127, tq = c >> 5, cc = c & 31;
          int pi = 0, el = 0, sh = 0;
#pragma unroll
          for (int p = 0; p < 16; p++) {
            const bool c4 = shared || BITS == 4;
            const int lo = c4 ? Codec<4>::lo(p) : Codec<BITS>::lo(p);
            const int hi = c4 ? Codec<4>::hi(p) : Codec<BITS>::hi(p);
            if (lo == cc) pi = p, el = 0, sh = c4 ? Codec<4>::slo(p) : Codec<BITS>::slo(p);
            if (hi == cc) pi = p, el = 1, sh = c4 ? Codec<4>::shi(p) : Codec<BITS>::shi(p);
          }
          const float hv = h * __uint_as_float((uint32_t)(127 - sh) << 23);  // h * 2^-sh, exact
          const uint32_t hi = f2bf(hv), lo = f2bf(hv - __uint_as_float(hi << 16));
          uint16_t *hb = P.hfrag + (size_t)d.slot * nblkI * 8 * 32 * 4;
          const int m = pi >> 1, reg = pi & 1;
          hb[(((blk * 8 + m) * 32 + 4 * b + tq) * 2 + reg) * 2 + el] = (uint16_t)hi;
          hb[(((blk * 8 + m) * 32 + 4 * (4 + b) + tq) * 2 + reg) * 2 + el] = (uint16_t)lo;
        }
        cta_signal(cnt + kCntGu + d.slot, 1u);
        if (q == 0) MOE_STAMP(13)
        if (q == s.nA + s.nB - 1) MOE_STAMP(14)
      } else {
        const int rt = d.row0 / 64;
        for (int j = tid; j < 64 * nb; j += NT) {
          const int r = j & 63, b = j >> 6;
          float y = 0.f;
          if (ok)
            for (int kb = 0; kb < nblkI; kb++) y += red[(kb * 8 + (r >> 3)) * 32 + (r & 7) * 4 + b];
          const float mb = shared ? gam[b] : wm[b * 64 + d.slot - s.hsi];
          P.ypart[((size_t)d.slot * 4 + b) * H + d.row0 + r] = mb * y;
        }
        __syncthreads();
        if (tid == 0) sflag[2] = atom_acq_rel_add(cnt + kCntDn + rt, 1u) == (unsigned)(s.nslots - 1);
        __syncthreads();
        if (sflag[2]) {
          // last unit of this 64-row range: sum the slots in a fixed order
          const int tpo = nb == 1 ? 8 : (nb == 2 ? 4 : 2);
          for (int j = tid; j < 64 * nb * tpo; j += NT) {
            const int o = j / tpo, part = j % tpo;
            const int r = o & 63, b = o >> 6;
            const float *yp = P.ypart + (size_t)b * H + d.row0 + r;
            float acc = 0.f;
#pragma unroll 4
            for (int sl = part; sl < s.nslots; sl += tpo) acc += __ldcg(yp + (size_t)sl * 4 * H);
            for (int off = tpo >> 1; off; off >>= 1) acc += __shfl_down_sync(FULL, acc, off, tpo);
            if (part == 0) {
              if (L.flags & kResidual) acc += __ldcg(src + (size_t)b * H + d.row0 + r);
              dst[(size_t)b * H + d.row0 + r] = acc;
            }
          }
          cta_signal(cnt + kCntRows, 1u);
        }
        __syncthreads();
        if (q == s.nA + s.nB) MOE_STAMP(15)
      }
    }
    qbase += (unsigned)n;
    MOE_STAMP(7)
#undef MOE_STAMP
  }
}

}  // namespace

static int fixed_smem(int H, int E, int bits) {
  const int nblkH = H / 128;
  const int E1 = (E + 1 + 3) & ~3;
  int b = 0;
  b += 4 * H * 4;                                  // xf
  b += nblkH * 256 * 8 * (bits == 4 ? 1 : 2);      // xa (+ xa4)
  b += 3 * 4 * (H / 64) * 4;                       // xs, cs, cs4
  b += 4 * E1 * 4;                                 // lg
  b += 2048 * 4;                                   // red
  b += (128 + 128 + 64 + 256 + 16) * 4;            // sidx sw uni wm gam+flags
  b += kMaxStages * 8;                             // barriers
  b += 64 * 8;                                     // slot -> record table
  b += kTscWords * 4;                              // transposed scales
  b += ((E + 1) & ~1) * 8;                         // expert addresses
  return b;
}

static int stage_bytes(int H, int I) {
  // the 4-bit tiles are the largest (the shared expert is always 4-bit)
  const int gu = 32 * code_pitch(H * 4 / 8, 4) + 64 * (H / 32);
  const int dn = 64 * code_pitch(I * 4 / 8, 4) + 128 * (I / 32);
  const int m = gu > dn ? gu : dn;
  return (m + 127) & ~127;
}

template <int BITS>
static int occupancy_t(int smem) {
  int n = 0;
  if (cudaFuncSetAttribute(decode_kernel<BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<BITS>, NT, smem) != cudaSuccess) return 0;
  return n;
}

int decode_plan(int device, FwdParams &p, int *grid, int *smem_bytes) {
  int sms = 0, optin = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess) return -1;
  const int fixed = fixed_smem(p.H, p.E, p.bits);
  const int sb = stage_bytes(p.H, p.I);
  int S = (optin - fixed) / sb;
  if (S > kMaxStages) S = kMaxStages;
  if (S < 1) return -1;
  p.stages = S;
  p.stage_bytes = sb;
  const int smem = fixed + S * sb;
  const int occ = p.bits == 4 ? occupancy_t<4>(smem) : p.bits == 3 ? occupancy_t<3>(smem) : occupancy_t<2>(smem);
  if (occ < 1) return -1;
  *grid = sms;
  *smem_bytes = smem;
  return 0;
}

template <int BITS>
static cudaError_t launch_t(const FwdParams &p, int grid, int smem, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_kernel<BITS>, p);
}

#ifdef MOE_DEBUG_CYCLES
extern "C" int moe_debug_cycles(long long *host64) {
  return (int)cudaMemcpyFromSymbol(host64, g_dbg_cycles, sizeof(long long) * 64);
}
#endif

cudaError_t launch_decode(const FwdParams &p, int grid, int smem, cudaStream_t st) {
  switch (p.bits) {
    case 4: return launch_t<4>(p, grid, smem, st);
    case 3: return launch_t<3>(p, grid, smem, st);
    case 2: return launch_t<2>(p, grid, smem, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
