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
//   G  gate_up units (internal slot, 16 gate rows + the matching 16 up rows):
//      codes stream from HBM straight into registers, are expanded to exact
//      bf16 integers and multiplied on the tensor cores against the staged
//      activations; scale and bias apply per 64-code group in fp32;
//      h = silu(gate) * up is written as bf16 hi/lo fragments for the down
//      projection.  A per-slot counter publishes completion.
//   D  down units (slot, 64 output rows): wait for the slot's h, multiply,
//      fold the routing weight (or the shared gate) into the result and store
//      a per-slot partial.  The last unit of a 64-row range (atomic ticket)
//      sums the slots in a fixed order, adds the residual and writes the
//      layer output.  No float atomics: results are bitwise reproducible.
// Every wait polls a counter with a deadline (%globaltimer); on expiry the
// kernel records MOE_ETIMEOUT and returns instead of hanging.
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
  if (threadIdx.x == 0) {
    bool ok = wait_geq(p, target, P);
    __threadfence();
    *flag = ok;
  }
  __syncthreads();
  const bool ok = *flag;
  __syncthreads();
  return ok;
}

__device__ void cta_signal(unsigned *p, unsigned v) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(p, v);
  }
}

// Activation fragments of one block of 128 positions for the codec whose pair
// table is (plo, phi): entry [blk][m][lane] holds the two bf16x2 A registers
// of MMA step m for lane (g, t): row g = hl*4 + b, value part hl (0 hi, 1 lo)
// of input row b, at positions 32t + pair code indices.
__device__ void stage_frags(const float *xf, int H, int nb, const int *plo, const int *phi, uint2 *xa) {
  const int nblk = H / 128;
  for (int e = threadIdx.x; e < nblk * 256; e += NT) {
    const int ln = e & 31, m = (e >> 5) & 7, blk = e >> 8;
    const int g = ln >> 2, t = ln & 3, hl = g >> 2, b = g & 3;
    uint32_t r0 = 0, r1 = 0;
    if (b < nb) {
      const float *base = xf + b * H + blk * 128 + 32 * t;
      r0 = split_part(base[plo[2 * m]], hl) | (split_part(base[phi[2 * m]], hl) << 16);
      r1 = split_part(base[plo[2 * m + 1]], hl) | (split_part(base[phi[2 * m + 1]], hl) << 16);
    }
    xa[e] = make_uint2(r0, r1);
  }
}

template <int B>
struct ItemRegs {
  uint32_t w[Codec<B>::kWords];
  uint32_t s0, s1, b0, b1;
};

// Load one item: codes of weight row (row0 + g) in block kb, and the scale /
// bias pairs (groups 2kb, 2kb+1) of rows row0 + 2t and row0 + 2t + 1.
template <int B>
__device__ __forceinline__ void load_item(ItemRegs<B> &it, const uint8_t *rec, const QOff &q, int inp,
                                          int row0, int kb, int g, int t) {
  const size_t rowbytes = (size_t)inp * B / 8;
  const uint8_t *cp = rec + q.w + (size_t)(row0 + g) * rowbytes + kb * (16 * B) + t * (4 * B);
  if constexpr (B == 4) {
    uint4 v = ldg_stream4(cp);
    it.w[0] = v.x, it.w[1] = v.y, it.w[2] = v.z, it.w[3] = v.w;
  } else if constexpr (B == 2) {
    uint2 v = ldg_stream2(cp);
    it.w[0] = v.x, it.w[1] = v.y;
  } else {
    it.w[0] = ldg_stream1(cp), it.w[1] = ldg_stream1(cp + 4), it.w[2] = ldg_stream1(cp + 8);
  }
  const size_t sp = (size_t)(inp / 64) * 2;
  const size_t r = (size_t)(row0 + 2 * t);
  it.s0 = ldg_stream1(rec + q.s + r * sp + kb * 4);
  it.s1 = ldg_stream1(rec + q.s + (r + 1) * sp + kb * 4);
  it.b0 = ldg_stream1(rec + q.b + r * sp + kb * 4);
  it.b1 = ldg_stream1(rec + q.b + (r + 1) * sp + kb * 4);
}

// One item on the tensor cores: 8 MMA steps over a block of 128 inputs for
// 8 weight rows, then per-group scale and bias in fp32.  Returns, in lanes
// 0..15 (b = lane/4), the results of rows 2t and 2t+1 of the item.
template <int B>
__device__ __forceinline__ void item_compute(const ItemRegs<B> &it, const uint2 (&a)[8], bool lowT, bool hl0,
                                             float xs0, float xs1, float mul, float &o0, float &o1) {
  uint32_t bf[16];
  Codec<B>::unpack(it.w, bf);
  float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int m = 0; m < 8; m++) {
    const uint32_t x0 = a[m].x, x1 = a[m].y;
    mma_bf16_16816(d, lowT ? x0 : 0u, lowT ? 0u : x0, lowT ? x1 : 0u, lowT ? 0u : x1, bf[2 * m], bf[2 * m + 1]);
  }
  float r0 = bf16lo(it.s0) * d[0] + bf16hi(it.s0) * d[2];
  float r1 = bf16lo(it.s1) * d[1] + bf16hi(it.s1) * d[3];
  if (hl0) {
    r0 += bf16lo(it.b0) * xs0 + bf16hi(it.b0) * xs1;
    r1 += bf16lo(it.b1) * xs0 + bf16hi(it.b1) * xs1;
  }
  r0 *= mul;
  r1 *= mul;
  o0 = r0 + __shfl_xor_sync(FULL, r0, 16);
  o1 = r1 + __shfl_xor_sync(FULL, r1, 16);
}

// items per warp: the smallest divisor of ntiles that covers all items
__device__ __forceinline__ int items_per_warp(int nitems, int ntiles) {
  const int need = (nitems + NW - 1) / NW;
  int ipw = 1;
  while (ipw < need) ipw *= 2;
  return ipw < ntiles ? ipw : ntiles;
}

// gate_up unit: rows [c0, c0+16) of the gate and [I+c0, I+c0+16) of the up
// projection, all H inputs.  Writes red[(kb*4 + nt)*32 + row*4 + b].
template <int B>
__device__ void gate_up_unit(const uint8_t *rec, const QOff &q, int H, int I, int c0, const uint2 *xa,
                             const float *xs, int nb, float *red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int nblk = H / 128, ntg = 4;
  const int nitems = nblk * ntg;
  const int ipw = items_per_warp(nitems, ntg);
  const int i0 = warp * ipw;
  if (i0 < nitems) {
    const int kb = i0 / ntg;
    ItemRegs<B> it[MAXIT];
#pragma unroll
    for (int k = 0; k < MAXIT; k++) {
      if (k < ipw) {
        const int nt = i0 % ntg + k;
        const int row0 = nt < 2 ? c0 + nt * 8 : I + c0 + (nt - 2) * 8;
        load_item<B>(it[k], rec, q, H, row0, kb, g, t);
      }
    }
    uint2 a[8];
#pragma unroll
    for (int m = 0; m < 8; m++) a[m] = xa[(kb * 8 + m) * 32 + lane];
    const int b = g & 3;
    const float xs0 = xs[b * (H / 64) + 2 * kb], xs1 = xs[b * (H / 64) + 2 * kb + 1];
#pragma unroll
    for (int k = 0; k < MAXIT; k++) {
      if (k < ipw) {
        float o0, o1;
        item_compute<B>(it[k], a, t < 2, g < 4, xs0, xs1, 1.f, o0, o1);
        const int nt = i0 % ntg + k;
        if (lane < 16 && b < nb) {
          red[(kb * ntg + nt) * 32 + (2 * t) * 4 + b] = o0;
          red[(kb * ntg + nt) * 32 + (2 * t + 1) * 4 + b] = o1;
        }
      }
    }
  }
}

// down unit: output rows [r0, r0+64) of one slot; A fragments of h come from
// the workspace.  mul[b] is the routing weight (or shared gate) of row b.
template <int B>
__device__ void down_unit(const uint8_t *rec, const QOff &q, int H, int I, int r0, const uint2 *hf,
                          const float *mul, int nb, float *red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int nblk = I / 128;
  const int nitems = nblk * 8;
  const int ipw = items_per_warp(nitems, 8);
  const int i0 = warp * ipw;
  if (i0 < nitems) {
    const int kb = i0 / 8;
    ItemRegs<B> it[MAXIT];
#pragma unroll
    for (int k = 0; k < MAXIT; k++) {
      if (k < ipw) load_item<B>(it[k], rec, q, I, r0 + (i0 % 8 + k) * 8, kb, g, t);
    }
    uint2 a[8];
    float hs = 0.f;
#pragma unroll
    for (int m = 0; m < 8; m++) {
      a[m] = __ldcg(hf + (kb * 8 + m) * 32 + lane);
      hs += bf16lo(a[m].x) + bf16hi(a[m].x) + bf16lo(a[m].y) + bf16hi(a[m].y);
    }
    // group sums of h: lanes t, t^1 share a group; add the lo part (g^4)
    hs += __shfl_xor_sync(FULL, hs, 1);
    hs += __shfl_xor_sync(FULL, hs, 16);
    const float other = __shfl_xor_sync(FULL, hs, 2);
    const float xs0 = t < 2 ? hs : other, xs1 = t < 2 ? other : hs;
    const int b = g & 3;
    const float mb = b < nb ? mul[b] : 0.f;
#pragma unroll
    for (int k = 0; k < MAXIT; k++) {
      if (k < ipw) {
        float o0, o1;
        item_compute<B>(it[k], a, t < 2, g < 4, xs0, xs1, mb, o0, o1);
        const int nt = i0 % 8 + k;
        if (lane < 16 && b < nb) {
          red[(kb * 8 + nt) * 32 + (2 * t) * 4 + b] = o0;
          red[(kb * 8 + nt) * 32 + (2 * t + 1) * 4 + b] = o1;
        }
      }
    }
  }
}

// Top-k of one row of E logits (ties to the lower id), then softmax over the
// k chosen.  Lane l holds ids [l*P, l*P+P).
__device__ void topk_warp(const float *lg, int E, int K, int *idx, float *w) {
  const int lane = threadIdx.x & 31;
  const int P = (E + 31) / 32;
  uint32_t taken = 0;
  for (int r = 0; r < K; r++) {
    uint32_t bk = 0;
    int bi = 0;
    for (int i = 0; i < P; i++) {
      const int e = lane * P + i;
      if (e < E && !((taken >> i) & 1u)) {
        const uint32_t key = orderable(lg[e]);
        if (key > bk) bk = key, bi = i;
      }
    }
    const uint32_t m = __reduce_max_sync(FULL, bk);
    const uint32_t bal = __ballot_sync(FULL, bk == m);
    const int wl = __ffs(bal) - 1;
    if (lane == wl) {
      taken |= 1u << bi;
      idx[r] = lane * P + bi;
      w[r] = lg[lane * P + bi];
    }
    __syncwarp();
  }
  const float mx = w[0];
  const float ev = lane < K ? expf(w[lane] - mx) : 0.f;
  const float z = warp_sum(ev);
  __syncwarp();
  if (lane < K) w[lane] = ev / z;
  __syncwarp();
}

// Union of the [nb][K] ids in first-seen order (warp 0).  Writes uni[],
// wm[b][slot] and returns U in *nu.  rk is 64 ints of scratch.
__device__ void union_warp(const int *sidx, const float *sw, int nb, int K, int *uni, float *wm, int *rk,
                           volatile int *nu) {
  const int lane = threadIdx.x & 31;
  const int n = nb * K;
  for (int j = lane; j < 256; j += 32) wm[j] = 0.f;
  int id[2], first[2], fpos[2];
#pragma unroll
  for (int h = 0; h < 2; h++) {
    const int pos = lane + 32 * h;
    id[h] = -1, first[h] = 0, fpos[h] = pos;
    if (pos < n) {
      id[h] = sidx[(pos / K) * 32 + pos % K];
      first[h] = 1;
      for (int j = 0; j < pos; j++) {
        if (sidx[(j / K) * 32 + j % K] == id[h]) {
          first[h] = 0;
          fpos[h] = j;
          break;
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
    const int pos = lane + 32 * h;
    if (pos < n) {
      const int slot = rk[fpos[h]];
      if (first[h]) uni[slot] = id[h];
      wm[(pos / K) * 64 + slot] = sw[(pos / K) * 32 + pos % K];
    }
  }
  if (lane == 0) *nu = __popc(b0) + __popc(b1);
  __syncwarp();
}

template <int BITS>
__global__ void __launch_bounds__(NT, 1) decode_kernel(const __grid_constant__ FwdParams P) {
  extern __shared__ __align__(16) unsigned char sm[];
  const int H = P.H, E = P.E, K = P.K, I = P.I, nb = P.nb;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int G = gridDim.x, cta = blockIdx.x;
  const int nblkH = H / 128, nblkI = I / 128;
  const int E1 = (E + 1 + 3) & ~3;
  const int ng = H / 64;

  float *xf = reinterpret_cast<float *>(sm);                 // [4][H]
  uint2 *xa = reinterpret_cast<uint2 *>(xf + 4 * H);         // [nblkH][8][32] routed codec order
  uint2 *xa4 = BITS == 4 ? xa : xa + nblkH * 256;            // shared (4-bit) order
  float *xs = reinterpret_cast<float *>(xa4 + nblkH * 256);  // [4][H/64]
  float *lg = xs + 4 * ng;                                   // [4][E1]
  float *red = lg + 4 * E1;                                  // [2048]
  int *sidx = reinterpret_cast<int *>(red + 2048);           // [4][32]
  float *sw = reinterpret_cast<float *>(sidx + 128);         // [4][32]
  int *uni = reinterpret_cast<int *>(sw + 128);              // [64]
  float *wm = reinterpret_cast<float *>(uni + 64);           // [4][64]
  float *gam = wm + 256;                                     // [4]
  volatile int *sflag = reinterpret_cast<volatile int *>(gam + 4);  // [16]
  int *ptab = const_cast<int *>(reinterpret_cast<volatile int *>(sflag + 16));  // [2 codecs][lo,hi][16]

  if (tid < 64) {
    const int which = tid >> 5, lohi = (tid >> 4) & 1, p = tid & 15;
    const int bits = which == 0 ? BITS : 4;
    ptab[tid] = lohi ? pair_hi(bits, p) : pair_lo(bits, p);
  }
  __syncthreads();
  const int *plo_r = ptab, *phi_r = ptab + 16, *plo_4 = ptab + 32, *phi_4 = ptab + 48;

  for (int l = 0; l < P.nl; l++) {
    const LayerP &L = P.L[l];
    unsigned *cnt = P.cnt + (size_t)l * kCntPerLayer;
    const bool hs = L.sgate != nullptr;
    const int hsi = hs ? 1 : 0;
    const float *src = l == 0 ? P.x : P.xbuf + (size_t)l * 4 * H;
    float *dst = l == P.nl - 1 ? P.out : P.xbuf + (size_t)(l + 1) * 4 * H;

    // ---- R: input, norm, fragments, router rows
    if (l > 0 && !cta_wait(P.cnt + (size_t)(l - 1) * kCntPerLayer + kCntRows, (unsigned)(H / 64), P, sflag))
      return;
    for (int i = tid; i < 4 * H; i += NT) xf[i] = i < nb * H ? __ldcg(src + i) : 0.f;
    __syncthreads();
    if (L.flags & kPrenorm) {
      if (warp < nb) {
        float ss = 0.f;
        for (int j = (tid & 31); j < H; j += 32) ss += xf[warp * H + j] * xf[warp * H + j];
        ss = warp_sum(ss);
        if ((tid & 31) == 0) red[warp] = 1.0f / sqrtf(ss / (float)H + 1e-6f);
      }
      __syncthreads();
      for (int i = tid; i < nb * H; i += NT) xf[i] *= red[i / H];
      __syncthreads();
    }
    stage_frags(xf, H, nb, plo_r, phi_r, xa);
    if (BITS != 4 && hs) stage_frags(xf, H, nb, plo_4, phi_4, xa4);
    for (int i = tid; i < 4 * ng; i += NT) {
      const float *p = xf + (i / ng) * H + (i % ng) * 64;
      float s = 0.f;
      for (int j = 0; j < 64; j++) s += p[j];
      xs[i] = s;
    }
    const int R = E + hsi;
    const int rr0 = (int)((long long)cta * R / G), rr1 = (int)((long long)(cta + 1) * R / G);
    const int nch = H / 256;
    const int nitem = (rr1 - rr0) * nch;
    __syncthreads();
    for (int it = warp; it < nitem; it += NW) {
      const int row = rr0 + it / nch, ch = it % nch, ln = tid & 31;
      const uint16_t *wrow = row < E ? L.router + (size_t)row * H : L.sgate;
      const uint4 wv = ldg_stream4(wrow + ch * 256 + ln * 8);
      const float wf[8] = {bf16lo(wv.x), bf16hi(wv.x), bf16lo(wv.y), bf16hi(wv.y),
                           bf16lo(wv.z), bf16hi(wv.z), bf16lo(wv.w), bf16hi(wv.w)};
      for (int b = 0; b < nb; b++) {
        const float *xp = xf + b * H + ch * 256 + ln * 8;
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < 8; j++) acc += wf[j] * xp[j];
        acc = warp_sum(acc);
        if (ln == 0) red[it * 4 + b] = acc;
      }
    }
    __syncthreads();
    for (int j = tid; j < (rr1 - rr0) * nb; j += NT) {
      const int r = j / nb, b = j % nb;
      float s = 0.f;
      for (int ch = 0; ch < nch; ch++) s += red[(r * nch + ch) * 4 + b];
      P.logits[((size_t)l * 4 + b) * (E + 1) + rr0 + r] = s;
    }
    if (rr1 > rr0) cta_signal(cnt + kCntRouter, (unsigned)(rr1 - rr0));

    // ---- T: top-k, softmax, union
    if (!cta_wait(cnt + kCntRouter, (unsigned)(R + (P.withhold ? 1 : 0)), P, sflag)) return;
    for (int i = tid; i < nb * (E + 1); i += NT) {
      const int b = i / (E + 1), e = i % (E + 1);
      lg[b * E1 + e] = e < R ? __ldcg(P.logits + ((size_t)l * 4 + b) * (E + 1) + e) : 0.f;
    }
    __syncthreads();
    if (warp < nb) topk_warp(lg + warp * E1, E, K, sidx + warp * 32, sw + warp * 32);
    if (tid < 4) gam[tid] = (hs && tid < nb) ? 1.f / (1.f + expf(-lg[tid * E1 + E])) : 0.f;
    __syncthreads();
    if (warp == 0) union_warp(sidx, sw, nb, K, uni, wm, reinterpret_cast<int *>(red), sflag + 1);
    __syncthreads();
    const int U = sflag[1];
    if (cta == 0) {
      if (P.slot_tab)
        for (int j = tid; j < kSlotStride; j += NT) {
          uint64_t v = j < U ? L.eaddr[uni[j]] : 0ull;
          if (j == kSlotStride - 2 || j == kSlotStride - 1) v = (uint64_t)U;
          P.slot_tab[(size_t)l * kSlotStride + j] = v;
        }
      if (P.wmap)
        for (int j = tid; j < kMaxNb * kSlotStride; j += NT) P.wmap[(size_t)l * kMaxNb * kSlotStride + j] = wm[j];
      if (P.topk_idx)
        for (int j = tid; j < nb * K; j += NT) P.topk_idx[(size_t)l * nb * K + j] = (uint32_t)sidx[(j / K) * 32 + j % K];
      if (P.topk_w)
        for (int j = tid; j < nb * K; j += NT) P.topk_w[(size_t)l * nb * K + j] = sw[(j / K) * 32 + j % K];
      if (P.logits_out)
        for (int j = tid; j < nb * E; j += NT) P.logits_out[j] = lg[(j / E) * E1 + j % E];
    }
    if (P.route_only) continue;

    // ---- G: gate_up units
    const int nslots = U + hsi;
    const int ups = I / 16;
    const int NU = nslots * ups;
    const int u0 = (int)((long long)cta * NU / G), u1 = (int)((long long)(cta + 1) * NU / G);
    for (int u = u0; u < u1; u++) {
      const int slot = u / ups, c0 = (u % ups) * 16;
      const bool shared = hs && slot == 0;
      const uint8_t *rec = shared ? L.srec : reinterpret_cast<const uint8_t *>(L.eaddr[uni[slot - hsi]]);
      const bool ok = rec != nullptr && ((uintptr_t)rec & 15u) == 0;
      if (!ok && tid == 0) atomicCAS(P.status, 0, kStatusDevice);
      if (ok) {
        if (shared)
          gate_up_unit<4>(rec, L.sgu, H, I, c0, xa4, xs, nb, red);
        else
          gate_up_unit<BITS>(rec, L.gu, H, I, c0, xa, xs, nb, red);
      }
      __syncthreads();
      // epilogue: h = silu(gate) * up for 16 rows x nb, scattered as bf16 hi/lo
      // A fragments in the order of this slot's down codec
      if (tid < 16 * nb) {
        const int i = tid & 15, b = tid >> 4;
        float gsum = 0.f, usum = 0.f;
        for (int kb = 0; kb < nblkH; kb++) {
          gsum += red[(kb * 4 + (i >> 3)) * 32 + (i & 7) * 4 + b];
          usum += red[(kb * 4 + 2 + (i >> 3)) * 32 + (i & 7) * 4 + b];
        }
        const float h = ok ? gsum / (1.f + expf(-gsum)) * usum : 0.f;
        const int pos = c0 + i;
        const int blk = pos >> 7, c = pos & 127, tq = c >> 5, cc = c & 31;
        const int *plo = shared ? plo_4 : plo_r, *phi = shared ? phi_4 : phi_r;
        int pi = 0, el = 0;
        for (int p = 0; p < 16; p++) {
          if (plo[p] == cc) pi = p, el = 0;
          if (phi[p] == cc) pi = p, el = 1;
        }
        const uint32_t hi = f2bf(h), lo = f2bf(h - __uint_as_float(hi << 16));
        uint16_t *hb = P.hfrag + (size_t)slot * nblkI * 8 * 32 * 4;
        const int m = pi >> 1, reg = pi & 1;
#pragma unroll
        for (int hl = 0; hl < 2; hl++) {
          const int ln = 4 * (hl * 4 + b) + tq;
          hb[(((blk * 8 + m) * 32 + ln) * 2 + reg) * 2 + el] = (uint16_t)(hl ? lo : hi);
        }
      }
      cta_signal(cnt + kCntGu + slot, 1u);
    }

    // ---- D: down units + finalisation
    const int nrt = H / 64;
    const int ND = nslots * nrt;
    const int d0 = (int)((long long)cta * ND / G), d1 = (int)((long long)(cta + 1) * ND / G);
    int cur = -1;
    for (int u = d0; u < d1; u++) {
      const int slot = u / nrt, rt = u % nrt;
      if (slot != cur) {
        if (!cta_wait(cnt + kCntGu + slot, (unsigned)ups, P, sflag)) return;
        cur = slot;
      }
      const bool shared = hs && slot == 0;
      const uint8_t *rec = shared ? L.srec : reinterpret_cast<const uint8_t *>(L.eaddr[uni[slot - hsi]]);
      const bool ok = rec != nullptr && ((uintptr_t)rec & 15u) == 0;
      float mul[4];
#pragma unroll
      for (int b = 0; b < 4; b++) mul[b] = shared ? gam[b] : wm[b * 64 + slot - hsi];
      const uint2 *hf = reinterpret_cast<const uint2 *>(P.hfrag + (size_t)slot * nblkI * 8 * 32 * 4);
      if (ok) {
        if (shared)
          down_unit<4>(rec, L.sdn, H, I, rt * 64, hf, mul, nb, red);
        else
          down_unit<BITS>(rec, L.dn, H, I, rt * 64, hf, mul, nb, red);
      }
      __syncthreads();
      for (int j = tid; j < 64 * nb; j += NT) {
        const int r = j & 63, b = j >> 6;
        float y = 0.f;
        if (ok)
          for (int kb = 0; kb < nblkI; kb++) y += red[(kb * 8 + (r >> 3)) * 32 + (r & 7) * 4 + b];
        P.ypart[((size_t)slot * 4 + b) * H + rt * 64 + r] = y;
      }
      __syncthreads();
      if (tid == 0) {
        __threadfence();
        const unsigned old = atomicAdd(cnt + kCntDn + rt, 1u);
        sflag[2] = old == (unsigned)(nslots - 1);
      }
      __syncthreads();
      if (sflag[2]) {
        __threadfence();
        for (int j = tid; j < 64 * nb; j += NT) {
          const int r = j & 63, b = j >> 6, o = rt * 64 + r;
          float s = 0.f;
          for (int sl = 0; sl < nslots; sl++) s += __ldcg(P.ypart + ((size_t)sl * 4 + b) * H + o);
          if (L.flags & kResidual) s += __ldcg(src + (size_t)b * H + o);
          dst[(size_t)b * H + o] = s;
        }
        cta_signal(cnt + kCntRows, 1u);
      }
      __syncthreads();
    }
  }
}

}  // namespace

int decode_smem_bytes(int H, int E, int bits) {
  const int nblkH = H / 128;
  const int E1 = (E + 1 + 3) & ~3;
  size_t b = 0;
  b += (size_t)4 * H * 4;                          // xf
  b += (size_t)nblkH * 256 * 8 * (bits == 4 ? 1 : 2);  // xa (+ xa4)
  b += (size_t)4 * (H / 64) * 4;                   // xs
  b += (size_t)4 * E1 * 4;                         // lg
  b += 2048 * 4;                                   // red
  b += (128 + 128 + 64 + 256 + 4 + 16 + 64) * 4;   // sidx sw uni wm gam sflag ptab
  return (int)b;
}

template <int BITS>
static cudaError_t launch_t(const FwdParams &p, int grid, cudaStream_t st) {
  const int smem = decode_smem_bytes(p.H, p.E, BITS);
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
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

cudaError_t launch_decode(const FwdParams &p, int grid, cudaStream_t st) {
  switch (p.bits) {
    case 4: return launch_t<4>(p, grid, st);
    case 3: return launch_t<3>(p, grid, st);
    case 2: return launch_t<2>(p, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

template <int BITS>
static int occupancy_t(int smem) {
  int n = 0;
  cudaFuncSetAttribute(decode_kernel<BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<BITS>, NT, smem) != cudaSuccess) return 0;
  return n;
}

// Grid of the cooperative launch: one CTA per SM (all co-resident).
int decode_grid(int device, int H, int E, int bits, int *grid) {
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return -1;
  const int smem = decode_smem_bytes(H, E, bits);
  const int occ = bits == 4 ? occupancy_t<4>(smem) : bits == 3 ? occupancy_t<3>(smem) : occupancy_t<2>(smem);
  if (occ < 1) return -1;
  *grid = sms;
  return 0;
}

}  // namespace moe
