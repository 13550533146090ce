// decode.cu -- persistent decode / speculative-verify kernel for nb <= 4 rows.
//
// One cooperative grid (one CTA per SM) runs every layer of a call.  Per layer:
//   R  each CTA loads the layer input (applying the unit RMSNorm when asked),
//      stages it as bf16 hi/lo tensor-core fragments, and computes its share of
//      the router rows (bf16 router x fp32 input on CUDA cores) plus the
//      shared-gate dot, each logit published as one 64-bit word that carries
//      its layer as a tag (a CTA's words sit together, one writer per line).
//   T  every CTA reads all logits in batches, then computes top-k, softmax and the
//      union itself (identical in every CTA, so no second grid-wide
//      handshake); CTA 0 publishes slot table, weight map and ids.
//   G  gate_up units (internal slot, 16 gate rows + the matching 16 up rows)
//   D  down units (slot, 64 output rows).
// Weight tiles of the units reach shared memory through bulk (TMA) copies
// into a ring of `stages` units, so HBM streams while the warps compute; two
// groups of eight warps (named barriers per group) each take the next unit
// not yet taken, and the group that frees a stage requests the unit `stages`
// places ahead.
// The shared expert's first gate_up units do not depend on routing and are
// requested before the layer input is even available.
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

#include <type_traits>

#include "codec.cuh"
#include "decode.cuh"

namespace moe {
namespace {

constexpr int NT = 512;
constexpr int NW = NT / 32;
constexpr int kProducerWarp = 1;  // warp (of the CTA, then of each unit group) that issues the bulk copies
// The weight units of a layer go to two groups of eight warps, each taking
// the next unit not yet taken (a shared-memory counter), so that one group's
// reductions, global writes and releases overlap the other group's
// tensor-core work and neither idles while units remain.
constexpr int kGroups = 2;
constexpr int GT = NT / kGroups;  // threads of a group
constexpr int GW = GT / 32;       // warps of a group

// Shared-memory row pitch of a staged code row of rb bytes (rows land
// contiguously: one bulk copy per block of rows).
__host__ __device__ constexpr int code_pitch(int rb, int) { return rb; }
constexpr unsigned FULL = 0xffffffffu;
constexpr uint32_t kResidual = 1, kPrenorm = 2, kLookahead = 4;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}

__device__ __forceinline__ uint32_t orderable(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// (a, b) -> bf16x2 hi = (bf16(a), bf16(b)) and lo = bf16 of the remainders (a first, low half)
__device__ __forceinline__ void split2(float a, float b, uint32_t &hi, uint32_t &lo) {
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(hi) : "f"(b), "f"(a));
  const float ra = a - __uint_as_float(hi << 16), rb = b - __uint_as_float(hi & 0xffff0000u);
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(lo) : "f"(rb), "f"(ra));
}

// floor(c*n/g); c*n stays far below 2^31 for every shape accepted
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

// Unit group g (threads GT*g .. GT*g+GT-1): barrier 1 + g, and the same with
// an AND over a predicate.
__device__ __forceinline__ void grp_sync(int g) { asm volatile("bar.sync %0, %1;" ::"r"(1 + g), "r"(GT) : "memory"); }
__device__ __forceinline__ bool grp_and(int g, bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n barrier.cta.red.and.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(1 + g), "r"(GT)
      : "memory");
  return r != 0;
}

// Group g: cta_wait / cta_signal for one unit group (gt: thread index in it).
__device__ bool grp_wait(const unsigned *p, unsigned target, const FwdParams &P, volatile int *flag, int g, int gt) {
  if (gt == 0) *flag = wait_geq(p, target, P);
  grp_sync(g);
  const bool ok = *flag;
  grp_sync(g);
  return ok;
}
__device__ void grp_signal(unsigned *p, unsigned v, int g, int gt) {
  grp_sync(g);
  if (gt == 0) red_release_add(p, v);
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
// (drain_stages: the same for the last unit issued into each stage.)
__device__ void drain_ring(uint64_t *bars, unsigned from, unsigned to, int S, const FwdParams &P) {
  if (threadIdx.x != 0) return;  // any one thread keeps the CTA (and its ring) alive until the copies land
  for (unsigned u = from; u < to; u++) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(&bars[u % S], (u / S) & 1u))
      if (globaltimer() - t0 > P.timeout_ns) return;
  }
}

__device__ void drain_stages(uint64_t *bars, const unsigned *last, int S, const FwdParams &P) {
  if (threadIdx.x != 0) return;
  for (int s = 0; s < S; s++) {
    if (last[s] == 0xffffffffu) continue;
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(&bars[s], (last[s] / S) & 1u))
      if (globaltimer() - t0 > P.timeout_ns) return;
  }
}

// ------------------------------------------------------------ activation staging
//
// MMA layout (m16n8k16, bf16 in, fp32 accumulate): A = 16 weight rows x 16
// k-slots of codes, B = 16 k-slots x 8 activation columns.  A block of 128
// inputs takes 8 MMA steps; lane (g, t) holds, for weight rows g and g+8, the
// 32 codes of quad position t (group t/2 of the block).  Column n of B is
// (group y = n/4, part hl = (n/2)&1 (bf16 hi or lo of the input), row bb = n&1)
// of activation rows b = 2*half + bb; B is zero where the k-slot belongs to
// the other group, so each column sums exactly one 64-code group.

// Thread pair (blk, t, b) turns the 32 inputs x[b][blk*128 + 32t .. +32) into
// the nonzero B registers of the lanes (col, t) with col in group t/2, for
// the 8 MMA steps (thread hh of the pair: steps 4hh .. 4hh+3), in codec B's
// pair order, each input pre-scaled by the 2^-s of its pair half (exact).
// Per 64-input group: xs = sum of x (bias term), cs = 128 * sum of 2^-s x
// (the offset the codes carry).  Rows b >= nb are never written here: their
// registers and sums stay at the zeros set when the kernel starts.
// Compact layout (the other group's zero columns are not stored):
// xb[blk][half][m][t][hl][bb], uint2 = k-slots (2t,2t+1), (2t+8,2t+9).
__device__ __forceinline__ int frag_index(int blk, int half, int m, int t, int hl, int bb) {
  return (((blk * 2 + half) * 8 + m) * 4 + t) * 4 + hl * 2 + bb;
}
template <int B>
__device__ void stage_frags(const float *xf, int H, int nb, uint2 *xb, float *xs, float *cs) {
  const int nblk = H / 128, per = nblk * 8, total = per * nb;
  const int lane = threadIdx.x & 31;
  // j = ((b * nblk + blk) * 4 + t) * 2 + hh; whole warps run each pass (shuffles)
  for (int j0 = (threadIdx.x & ~31); j0 < total; j0 += NT) {
    const int j = j0 + lane;
    const bool valid = j < total;
    int b = 0, jj = valid ? j : 0;
    while (jj >= per) jj -= per, b++;
    const int hh = jj & 1, t = (jj >> 1) & 3, blk = jj >> 3;
    const int half = b >> 1, bb = b & 1;
    float v[32];
    const float4 *src = reinterpret_cast<const float4 *>(xf + b * H + blk * 128 + 32 * t);
#pragma unroll
    for (int i = 0; i < 8; i++) {
      const float4 q = valid ? src[i] : make_float4(0.f, 0.f, 0.f, 0.f);
      v[4 * i] = q.x, v[4 * i + 1] = q.y, v[4 * i + 2] = q.z, v[4 * i + 3] = q.w;
    }
    float sx = 0.f, sc = 0.f;
#pragma unroll
    for (int i = 0; i < 16; i++) sx += hh ? v[16 + i] : v[i];
#pragma unroll
    for (int mq = 0; mq < 4; mq++) {
      const int m = 4 * hh + mq;
      float a[4];
#pragma unroll
      for (int hm = 0; hm < 2; hm++) {  // this thread's half selects the pairs at compile time per branch
#pragma unroll
        for (int k = 0; k < 2; k++) {
          const int p = 2 * (4 * hm + mq) + k;
          if (hm == hh) {
            a[2 * k] = v[Codec<B>::lo(p)] * pow2neg(Codec<B>::slo(p));
            a[2 * k + 1] = v[Codec<B>::hi(p)] * pow2neg(Codec<B>::shi(p));
          }
        }
      }
      uint32_t hi0, lo0, hi1, lo1;
      split2(a[0], a[1], hi0, lo0);
      split2(a[2], a[3], hi1, lo1);
      // the offset sum from exactly the values the MMA sees (hi + lo), so the
      // 128 offset cancels without amplifying the split's residual
      sc += (bf16lo(hi0) + bf16lo(lo0)) + (bf16hi(hi0) + bf16hi(lo0)) + (bf16lo(hi1) + bf16lo(lo1)) +
            (bf16hi(hi1) + bf16hi(lo1));
      if (valid) {
        xb[frag_index(blk, half, m, t, 0, bb)] = make_uint2(hi0, hi1);
        xb[frag_index(blk, half, m, t, 1, bb)] = make_uint2(lo0, lo1);
      }
    }
    // the pair (hh), then the two quad positions of the group (t, t ^ 1)
    sx += __shfl_xor_sync(FULL, sx, 1);
    sc += __shfl_xor_sync(FULL, sc, 1);
    sx += __shfl_xor_sync(FULL, sx, 2);
    sc += __shfl_xor_sync(FULL, sc, 2);
    if (valid && hh == 0 && (t & 1) == 0) {
      const int y = t >> 1;
      if (xs) xs[b * (H / 64) + 2 * blk + y] = sx;
      cs[b * (H / 64) + 2 * blk + y] = 128.f * sc;
    }
  }
}

// ------------------------------------------------------------ tensor-core items

// Column-pair constants of one lane for one half of the activation rows:
// accumulator start (minus the offset sum of the lane's group on hi-part
// columns, 0 on lo-part ones) and the group's input sums (hi-part columns
// only, so the bias enters once).
struct ColC {
  float c0, c1, x0, x1;
};

// One item: 16 weight rows (stage rows r0 .. r0+15) x one block of 128
// inputs, for nh halves of the activation rows.  Codes come from the stage;
// sc / bi point at the scale / bias pair word of row r0 for this block, the
// words of the next rows `ss` words apart (the stage's [row][pair] tables).  Returns per lane (t == 0 lanes after the sums) the outputs of rows
// g and g+8 for activation rows b = 2*half + {0,1}.
template <int B, int NH, bool O4 = false>
__device__ __forceinline__ void item_compute(const uint8_t *row_g, const uint8_t *row_g8, const uint32_t *sc,
                                             const uint32_t *bi, int ss, int g, int y, const uint2 (&xb)[NH][8],
                                             const ColC (&cc)[NH], float (&o)[NH][4]) {
  // O4: the 4-bit pair order for every width (a union mixing widths)
  using C = typename std::conditional<O4, CodecO4<B>, Codec<B>>::type;
  uint32_t wa[C::kWords], wb[C::kWords];
  if constexpr (B == 4) {
    const uint4 va = *reinterpret_cast<const uint4 *>(row_g), vb = *reinterpret_cast<const uint4 *>(row_g8);
    wa[0] = va.x, wa[1] = va.y, wa[2] = va.z, wa[3] = va.w;
    wb[0] = vb.x, wb[1] = vb.y, wb[2] = vb.z, wb[3] = vb.w;
  } else if constexpr (B == 2) {
    const uint2 va = *reinterpret_cast<const uint2 *>(row_g), vb = *reinterpret_cast<const uint2 *>(row_g8);
    wa[0] = va.x, wa[1] = va.y, wb[0] = vb.x, wb[1] = vb.y;
  } else {
    const uint32_t *pa = reinterpret_cast<const uint32_t *>(row_g), *pb = reinterpret_cast<const uint32_t *>(row_g8);
    wa[0] = pa[0], wa[1] = pa[1], wa[2] = pa[2], wb[0] = pb[0], wb[1] = pb[1], wb[2] = pb[2];
  }
  const uint32_t sg = sc[g * ss], sg8 = sc[(g + 8) * ss], bg = bi[g * ss], bg8 = bi[(g + 8) * ss];
  uint32_t fa[16], fb[16];
  C::unpack(wa, fa);
  C::unpack(wb, fb);
  const float s0 = y ? bf16hi(sg) : bf16lo(sg), s8 = y ? bf16hi(sg8) : bf16lo(sg8);
  const float b0 = y ? bf16hi(bg) : bf16lo(bg), b8 = y ? bf16hi(bg8) : bf16lo(bg8);
#pragma unroll
  for (int h = 0; h < NH; h++) {
    float d[4] = {cc[h].c0, cc[h].c1, cc[h].c0, cc[h].c1}, e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int m = 0; m < 8; m += 2) {
      mma_bf16_16816(d, fa[2 * m], fb[2 * m], fa[2 * m + 1], fb[2 * m + 1], xb[h][m].x, xb[h][m].y);
      mma_bf16_16816(e, fa[2 * m + 2], fb[2 * m + 2], fa[2 * m + 3], fb[2 * m + 3], xb[h][m + 1].x, xb[h][m + 1].y);
    }
    float r0 = s0 * (d[0] + e[0]) + b0 * cc[h].x0;
    float r1 = s0 * (d[1] + e[1]) + b0 * cc[h].x1;
    float r2 = s8 * (d[2] + e[2]) + b8 * cc[h].x0;
    float r3 = s8 * (d[3] + e[3]) + b8 * cc[h].x1;
    // sum over the quad: parts hi / lo (t, t^1) and the two groups (t, t^2)
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
      r0 += __shfl_xor_sync(FULL, r0, off);
      r1 += __shfl_xor_sync(FULL, r1, off);
      r2 += __shfl_xor_sync(FULL, r2, off);
      r3 += __shfl_xor_sync(FULL, r3, off);
    }
    o[h][0] = r0, o[h][1] = r1, o[h][2] = r2, o[h][3] = r3;
  }
}

// B registers of lane (g, t) for one block and half: its column's entry if
// the column belongs to the lane's group, else zero.
template <int NH>
__device__ __forceinline__ void load_bfrag(const uint2 *xb, int blk, int lane, uint2 (&x)[NH][8]) {
  const int g = lane >> 2, t = lane & 3;
  const bool mine = (g >> 2) == (t >> 1);
#pragma unroll
  for (int h = 0; h < NH; h++)
#pragma unroll
    for (int m = 0; m < 8; m++) {
      const uint2 v = xb[frag_index(blk, h, m, t, (g >> 1) & 1, g & 1)];
      x[h][m] = mine ? v : make_uint2(0u, 0u);
    }
}

// Column constants of lane (g, t) for one half from the group sums of
// activation rows b = 2*half, 2*half+1 (xs: input sums, cs: offset sums).
__device__ __forceinline__ ColC col_consts(float cs0, float cs1, float xs0, float xs1, bool hipart) {
  ColC c;
  c.c0 = hipart ? -cs0 : 0.f, c.c1 = hipart ? -cs1 : 0.f;
  c.x0 = hipart ? xs0 : 0.f, c.x1 = hipart ? xs1 : 0.f;
  return c;
}

// Items of a gate_up unit: (block kb, row tile 0 = the 16 gate rows, 1 = the
// 16 up rows).  sw: the unit's scale words [32][H/128], then its bias words.
// Writes red[(kb*2 + tile)*64 + row*4 + b].
// Warp wi of nw takes blocks wi, wi + nw, ... (both tiles of a block share
// its activation registers).
template <int B, int NH, bool O4 = false>
__device__ void gate_up_compute(const uint8_t *st, const uint32_t *sw, int H, const uint2 *xb, const float *xs,
                                const float *cs, int nb, float *red, int wi, int nw) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3, y = t >> 1;
  const int nblk = H / 128;
  const int rb = H * B / 8, np = H / 128, ng = H / 64;
#pragma unroll 1
  for (int kb = wi; kb < nblk; kb += nw) {
  uint2 x[NH][8];
  ColC cc[NH];
  load_bfrag<NH>(xb, kb, lane, x);
#pragma unroll
  for (int h = 0; h < NH; h++) {
    const int b0 = 2 * h, b1 = 2 * h + 1, grp = 2 * kb + y;
    cc[h] = col_consts(cs[b0 * ng + grp], cs[b1 * ng + grp], xs[b0 * ng + grp], xs[b1 * ng + grp], (t & 1) == 0);
  }
  const uint32_t *sc = sw + kb, *bi = sw + 32 * np + kb;
#pragma unroll 1
  for (int tile = 0; tile < 2; tile++) {
    const int r0 = 16 * tile;
    float o[NH][4];
    item_compute<B, NH, O4>(st + (r0 + g) * rb + kb * (16 * B) + t * (4 * B),
                        st + (r0 + g + 8) * rb + kb * (16 * B) + t * (4 * B), sc + r0 * np, bi + r0 * np, np, g, y,
                        x, cc, o);
    if (t == 0) {
      float *rp = red + (kb * 2 + tile) * 64;
#pragma unroll
      for (int h = 0; h < NH; h++) {
        *reinterpret_cast<float2 *>(rp + g * 4 + 2 * h) = make_float2(o[h][0], o[h][1]);
        *reinterpret_cast<float2 *>(rp + (g + 8) * 4 + 2 * h) = make_float2(o[h][2], o[h][3]);
      }
    }
  }
  }
}

// Items of a down unit: (block kb, row tile of 16 of the unit's 64 output
// rows).  xb / xs / cs: the slot's h fragments and group sums, staged in
// shared memory.  sw: the unit's scale words [64][I/128], then its bias
// words.  Writes red[(kb*4 + tile)*64 + row*4 + b].
// Warp wi of nw takes passes wi, wi + nw, ... of two row tiles of one
// block (pass p: block p / 2, tiles 2 (p % 2) and 2 (p % 2) + 1).
template <int B, int NH, bool O4 = false>
__device__ void down_compute(const uint8_t *st, const uint32_t *sw, int I, const uint2 *xb, const float *xs,
                             const float *cs, int nb, float *red, int wi, int nw) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3, y = t >> 1;
  const int npass = (I / 128) * 2;
  const int rb = I * B / 8, np = I / 128, ng = I / 64;
#pragma unroll 1
  for (int pass = wi; pass < npass; pass += nw) {
  const int kb = pass >> 1;
  uint2 x[NH][8];
  ColC cc[NH];
  load_bfrag<NH>(xb, kb, lane, x);
#pragma unroll
  for (int h = 0; h < NH; h++) {
    const int b0 = 2 * h, b1 = 2 * h + 1, grp = 2 * kb + y;
    cc[h] = col_consts(cs[b0 * ng + grp], cs[b1 * ng + grp], xs[b0 * ng + grp], xs[b1 * ng + grp], (t & 1) == 0);
  }
  const uint32_t *sc = sw + kb, *bi = sw + 64 * np + kb;
#pragma unroll 1
  for (int k = 0; k < 2; k++) {
    const int tile = 2 * (pass & 1) + k;
    const int r0 = 16 * tile;
    float o[NH][4];
    item_compute<B, NH, O4>(st + (r0 + g) * rb + kb * (16 * B) + t * (4 * B),
                        st + (r0 + g + 8) * rb + kb * (16 * B) + t * (4 * B), sc + r0 * np, bi + r0 * np, np, g, y,
                        x, cc, o);
    if (t == 0) {
      float *rp = red + (kb * 4 + tile) * 64;
#pragma unroll
      for (int h = 0; h < NH; h++) {
        *reinterpret_cast<float2 *>(rp + g * 4 + 2 * h) = make_float2(o[h][0], o[h][1]);
        *reinterpret_cast<float2 *>(rp + (g + 8) * 4 + 2 * h) = make_float2(o[h][2], o[h][3]);
      }
    }
  }
  }
}

// One unit group (g; gt: thread index in it): bring one slot's h fragments
// into shared memory and form its per-group sums: hxs = sum of h (bias term), hcs = 128 * sum of 2^-s h as the
// MMA sees it (offset), [b][I/64].  Codec C is the slot's down codec.
template <int C>
__device__ void stage_h(const uint2 *hf, int I, int nb, uint2 *hsm, float *hxs, float *hcs, int g, int gt) {
  const int nblk = I / 128;
  const int n = nblk * 256;
  for (int i = gt; i < n; i += GT) hsm[i] = __ldcg(hf + i);
  grp_sync(g);
  // thread (kb, y, b, part): 4 of the 32 entries (t in {2y, 2y+1}, m, hl) of a group
  const int ng = I / 64;
  for (int j = gt; j < nblk * 64; j += GT) {
    const int part = j & 7, b = (j >> 3) & 3, y = (j >> 5) & 1, kb = j >> 6;
    float ssc = 0.f, sun = 0.f;
    if (b < nb) {
#pragma unroll
      for (int k = 0; k < 4; k++) {
        const int e = part * 4 + k;  // e = (t - 2y) * 16 + m * 2 + hl
        const int tt = 2 * y + (e >> 4), m = (e >> 1) & 7, hl = e & 1;
        const uint2 v = hsm[frag_index(kb, b >> 1, m, tt, hl, b & 1)];
        const float v0 = bf16lo(v.x), v1 = bf16hi(v.x), v2 = bf16lo(v.y), v3 = bf16hi(v.y);
        ssc += v0 + v1 + v2 + v3;
        float w0 = 1.f, w1 = 1.f, w2 = 1.f, w3 = 1.f;
        if (C != 4) {
#pragma unroll
          for (int mm = 0; mm < 8; mm++)
            if (mm == m) {
              w0 = (float)(1 << Codec<C>::slo(2 * mm)), w1 = (float)(1 << Codec<C>::shi(2 * mm));
              w2 = (float)(1 << Codec<C>::slo(2 * mm + 1)), w3 = (float)(1 << Codec<C>::shi(2 * mm + 1));
            }
        }
        sun += v0 * w0 + v1 * w1 + v2 * w2 + v3 * w3;
      }
    }
#pragma unroll
    for (int o = 4; o; o >>= 1) {
      ssc += __shfl_xor_sync(FULL, ssc, o);
      sun += __shfl_xor_sync(FULL, sun, o);
    }
    if (part == 0) {
      hcs[b * ng + 2 * kb + y] = 128.f * ssc;
      hxs[b * ng + 2 * kb + y] = sun;
    }
  }
}

// ------------------------------------------------------------ routing

// Top-k of one row of E <= 1024 logits (ties to the lower id), then softmax
// over the k chosen.  Lane l holds ids l, l + 32, ... as order-preserving
// keys in registers; each round one warp max finds the largest key and one
// warp min the lowest id holding it; the winner's lane rescans its keys, and
// lane r keeps the r-th winner, so nothing is written until the end.
template <int PM>
__device__ void topk_warp(const float *lg, int E, int K, int *idx, float *w) {
  const int lane = threadIdx.x & 31;
  uint32_t key[PM];
#pragma unroll
  for (int i = 0; i < PM; i++) {
    const int e = i * 32 + lane;
    key[i] = e < E ? orderable(lg[e]) : 0u;
  }
  uint32_t bk = 0;
  int bi = 0;
#pragma unroll
  for (int i = 0; i < PM; i++)
    if (key[i] > bk) bk = key[i], bi = i;
  int myid = 0;
#pragma unroll 1
  for (int r = 0; r < K; r++) {
    const uint32_t m = __reduce_max_sync(FULL, bk);
    const uint32_t id = __reduce_min_sync(FULL, bk == m ? (uint32_t)(bi * 32 + lane) : 0xffffffffu);
    if (lane == r) myid = (int)id;
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
  const float myl = lane < K ? lg[myid] : 0.f;
  const float mx = __shfl_sync(FULL, myl, 0);
  const float ev = lane < K ? expf(myl - mx) : 0.f;
  const float z = warp_sum(ev);
  if (lane < K) idx[lane] = myid, w[lane] = ev / z;
  __syncwarp();
}

// Union of the [nb][K] ids in first-seen order (warp 0).  Writes uni[],
// wm[b][slot] and *nu = U.  posof[E] holds INT_MAX on entry and on exit; rk
// is 64 ints of scratch.  Position p = b*K + r: each position records itself
// in posof[id] by an atomic min, so the first occurrence of every id is the
// position that survives; firsts are ranked by a ballot.
__device__ void union_warp(const int *sidx, const float *sw, int nb, int K, int *uni, float *wm, int *posof, int *rk,
                           volatile int *nu) {
  const int lane = threadIdx.x & 31;
  for (int j = lane; j < 256; j += 32) wm[j] = 0.f;
  if (nb == 1) {  // one row: its k ids are distinct, in rank order
    __syncwarp();
    if (lane < K) uni[lane] = sidx[lane], wm[lane] = sw[lane];
    if (lane == 0) *nu = K;
    __syncwarp();
    return;
  }
  const int n = nb * K;
  int id[2], pb[2], pr[2];
#pragma unroll
  for (int h = 0; h < 2; h++) {
    const int p = lane + 32 * h;
    pb[h] = p / K, pr[h] = p - (p / K) * K;
    id[h] = p < n ? sidx[pb[h] * 32 + pr[h]] : -1;
    if (p < n) atomicMin(&posof[id[h]], p);
  }
  __syncwarp();
  bool first[2];
#pragma unroll
  for (int h = 0; h < 2; h++) first[h] = lane + 32 * h < n && posof[id[h]] == lane + 32 * h;
  const uint32_t b0 = __ballot_sync(FULL, first[0]), b1 = __ballot_sync(FULL, first[1]);
  const uint32_t lt = (1u << lane) - 1u;
  if (first[0]) rk[lane] = __popc(b0 & lt);
  if (first[1]) rk[lane + 32] = __popc(b0) + __popc(b1 & lt);
  __syncwarp();
#pragma unroll
  for (int h = 0; h < 2; h++) {
    if (lane + 32 * h < n) {
      const int slot = rk[posof[id[h]]];
      if (first[h]) uni[slot] = id[h];
      wm[pb[h] * 64 + slot] = sw[pb[h] * 32 + pr[h]];
    }
  }
  __syncwarp();
#pragma unroll
  for (int h = 0; h < 2; h++)
    if (lane + 32 * h < n) posof[id[h]] = 0x7fffffff;
  if (lane == 0) *nu = __popc(b0) + __popc(b1);
  __syncwarp();
}

// The union's slots this GPU computes, in union order within each tier:
// records in device memory first, then records in host memory.  An expert
// whose record is not on this GPU at all (address 0: an expert-parallel
// shard holds only its own experts) is left out, and so is a host-memory
// one whose weight is below cut_w in every row (the deadline cut of weak
// experts).  wm columns move with their slots; tier_out[j] = 1 for a kept
// host-memory slot j.  nkeep[0] = slots kept, nkeep[1] = of them in device
// memory.  (warp 0; et_s may be null: every record in device memory)
__device__ __forceinline__ void place_union(int *uni, float *wm, const uint64_t *eaddr_s, const uint8_t *et_s, float cut_w, int U,
                            int *tier_out, volatile int *nkeep) {
  const int lane = threadIdx.x & 31;
  int id[2];
  bool dev[2], hst[2];
  float w[2][4];
#pragma unroll
  for (int h = 0; h < 2; h++) {
    const int j = lane + 32 * h;
    id[h] = j < U ? uni[j] : 0;
    float wmax = 0.f;
#pragma unroll
    for (int b = 0; b < 4; b++) w[h][b] = wm[b * 64 + j], wmax = fmaxf(wmax, w[h][b]);
    const bool here = j < U && eaddr_s[id[h]] != 0ull;
    const bool host = et_s != nullptr && et_s[id[h]] != 0;
    dev[h] = here && !host;
    hst[h] = here && host && !(wmax < cut_w);
  }
  const uint32_t bd0 = __ballot_sync(FULL, dev[0]), bd1 = __ballot_sync(FULL, dev[1]);
  const uint32_t bh0 = __ballot_sync(FULL, hst[0]), bh1 = __ballot_sync(FULL, hst[1]);
  const uint32_t lt = (1u << lane) - 1u;
  const int nd = __popc(bd0) + __popc(bd1);
  __syncwarp();
#pragma unroll
  for (int h = 0; h < 2; h++)
#pragma unroll
    for (int b = 0; b < 4; b++) wm[b * 64 + lane + 32 * h] = 0.f;
  __syncwarp();
#pragma unroll
  for (int h = 0; h < 2; h++) {
    if (dev[h] || hst[h]) {
      const int pos = dev[h] ? (h == 0 ? __popc(bd0 & lt) : __popc(bd0) + __popc(bd1 & lt))
                             : nd + (h == 0 ? __popc(bh0 & lt) : __popc(bh0) + __popc(bh1 & lt));
      uni[pos] = id[h];
      tier_out[pos] = hst[h] ? 1 : 0;
#pragma unroll
      for (int b = 0; b < 4; b++) wm[b * 64 + pos] = w[h][b];
    }
  }
  if (lane == 0) nkeep[0] = nd + __popc(bh0) + __popc(bh1), nkeep[1] = nd;
  __syncwarp();
}

// Every CTA's published logits into lg[b][e]: word (c, j) of writer CTA c
// in buf holds logit row rr0(c) + j / nb (rows split over the CTAs as
// fdiv_mul(c, Rl, G)) of activation row j % nb, tagged `tag`.  A word with
// another tag is waited out; a wait that runs out reports a timeout, or with
// `hint` (the lookahead prediction) only makes the call return false after
// kHintWaitNs.  Batches of four words: every load of a batch first, then the
// tags.  (Out of line: its temporaries stay out of the unit loop's registers.)
constexpr uint64_t kHintWaitNs = 20000;
__device__ __noinline__ bool read_tagged(const FwdParams &P, const unsigned long long *buf, unsigned tag, int Rl,
                                         int E1, float *lg, bool hint) {
  const int tid = threadIdx.x, G = gridDim.x, nb = P.nb;
  bool ok = true;
  const int per = ((Rl + G - 1) / G) * nb, total = G * per;
  for (int t0 = tid; t0 < total; t0 += 4 * NT) {
    unsigned long long w[4];
    int word[4], dst[4];
#pragma unroll
    for (int k = 0; k < 4; k++) {
      const int t = t0 + k * NT;
      word[k] = -1;
      if (t < total) {
        const int c = t / per, j = t - c * per;
        const int c0 = fdiv_mul(c, Rl, G), c1 = fdiv_mul(c + 1, Rl, G);
        if (j < (c1 - c0) * nb) {
          word[k] = c * kLogitWords + j;
          dst[k] = (j % nb) * E1 + c0 + j / nb;
          w[k] = ld_relaxed_u64(buf + word[k]);
        }
      }
    }
#pragma unroll
    for (int k = 0; k < 4; k++) {
      if (word[k] < 0 || !ok) continue;
      if ((unsigned)(w[k] >> 32) != tag) {
        const uint64_t t0w = globaltimer();
        unsigned spins = 0;
        while ((unsigned)((w[k] = ld_relaxed_u64(buf + word[k])) >> 32) != tag) {
          if ((++spins & 15u) == 0) {
            if (ld_volatile_int(P.status) != 0) {
              ok = false;
              break;
            }
            if (globaltimer() - t0w > (hint ? kHintWaitNs : P.timeout_ns)) {
              if (!hint) atomicCAS(P.status, 0, kStatusTimeout);
              ok = false;
              break;
            }
          }
        }
      }
      lg[dst[k]] = __uint_as_float((uint32_t)w[k]);
    }
  }
  return ok;
}


// Layer l's logits: tag l + 1, in the half of the buffer for l's parity.
// The half cannot be rewritten under a reader: layer l + 2's rows are
// written only after layer l + 1 has finished, which needs every CTA's layer
// l + 1 router rows, which each CTA writes after it has read layer l's.
// (The lookahead's logits for layer l + 1, tag l + 2, use a buffer of their
// own on the same parity rule.)
__device__ __noinline__ bool read_logits(const FwdParams &P, int l, int Rl, int E1, float *lg) {
  return read_tagged(P, P.lgw + (size_t)(l & 1) * kMaxGrid * kLogitWords, (unsigned)l + 1u, Rl, E1, lg, false);
}

// ------------------------------------------------------------ unit schedule

// The layer's gate_up units form one list, slot by slot (the shared expert's
// first), and so do its down units; CTA c takes list entries c, c + G,
// c + 2G, ... of each (G = grid size).  A slot's units then sit in the same
// position of consecutive CTAs, so slots complete in waves and the first
// down units find their h ready early.  The shared expert's gate_up units are
// known before routing (nA of this CTA's first units).
struct Sched {
  int hsi, ups, nrt, U, nslots;
  int nA;    // this CTA's shared gate_up units (requested before routing)
  int nGU;   // this CTA's gate_up units (shared + routed)
  int nD;    // this CTA's down units
  __device__ int n() const { return nGU + nD; }
};

// entries c, c + G, ... of a list of T
__device__ __forceinline__ int rr_count(int c, int T, int G) { return T > c ? (T - c + G - 1) / G : 0; }

struct UnitDesc {
  int down, slot, row0;  // row0: gate_up chunk start (inter rows) or down output row start
  const uint8_t *rec;
  QOff q;
  int bits;
  int host;  // the record is in host memory: its tile is read by the computing group, not bulk-copied
};

// BITS = 0: a union mixing widths; slot j's width is sbits[j].  stier[j]:
// slot j's record is in host memory.
template <int BITS>
__device__ __forceinline__ UnitDesc get_unit(int q, const Sched &s, const LayerP &L,
                                             const uint8_t *const *rect, const int *sbits, const int *stier) {
  UnitDesc d;
  const int c = blockIdx.x, G = gridDim.x;
  if (q < s.nGU) {
    const int u = c + q * G;  // entry of the gate_up list
    d.down = 0, d.slot = u / s.ups, d.row0 = (u % s.ups) * 16;
  } else {
    const int v = c + (q - s.nGU) * G;  // entry of the down list
    d.down = 1, d.slot = v / s.nrt, d.row0 = (v % s.nrt) * 64;
  }
  const bool shared = s.hsi && d.slot == 0;
  d.rec = shared ? L.srec : rect[d.slot];
  d.host = shared ? 0 : stier[d.slot];
  if (BITS == 0 && !shared) {
    d.bits = sbits[d.slot];
    d.q = d.down ? L.dnw[4 - d.bits] : L.guw[4 - d.bits];
  } else {
    d.q = shared ? (d.down ? L.sdn : L.sgu) : (d.down ? L.dn : L.gu);
    d.bits = shared ? 4 : BITS;
  }
  return d;
}

// Producer warp: request the weight tile of one unit into its ring stage:
// the code rows (gate_up: 16 gate rows then the matching 16 up rows; down:
// 64 output rows), then their scales, then their biases, row-major.
// host_fill: this stage's word, 1 while its last fill was by cp.async.
__device__ void issue_unit(const UnitDesc &d, int H, int I, uint8_t *st, uint64_t *bar, int *status,
                           unsigned *host_fill) {
  const int lane = threadIdx.x & 31;
  const bool ok = d.rec != nullptr && ((uintptr_t)d.rec & 15u) == 0;
  if (ok && d.host) {
    // a record in host memory: the warp's lanes read the tile over the C2C
    // link with 16-byte cp.async copies (the ordinary load path), in the
    // layout the bulk copies below give (code rows, then scale rows, then
    // bias rows; gate_up: the gate then the up half of each; every segment
    // a whole number of 16-byte pieces), each lane's copies registered on
    // the stage barrier; lane 0 then makes the phase's one arrival
    const int inp = d.down ? I : H, nrow = d.down ? 64 : 16, rows = d.down ? 64 : 32;
    const uint32_t rb = inp * d.bits / 8, sp = inp / 32;
    for (int k = 0; k < (d.down ? 3 : 6); k++) {
      const int kind = d.down ? k : k >> 1, half = d.down ? 0 : k & 1;
      const uint32_t rowb = kind == 0 ? rb : sp;
      const uint8_t *src =
          d.rec + (kind == 0 ? d.q.w : kind == 1 ? d.q.s : d.q.b) + (size_t)(d.row0 + half * I) * rowb;
      uint8_t *dst = kind == 0 ? st + half * nrow * rb : st + rows * rb + (kind - 1) * rows * sp + half * nrow * sp;
      const int n = (int)((nrow * rowb) >> 4);
      for (int i = lane; i < n; i += 32) cp_async16(dst + 16 * i, src + 16 * i);
    }
    cp_async_mbar_arrive(bar);
    __syncwarp();
    if (lane == 0) *host_fill = 1u, mbar_arrive(bar);
    return;
  }
  if (lane != 0) return;
  if (!ok) {
    atomicCAS(status, 0, kStatusDevice);
    mbar_expect_tx(bar, 0);  // completes the phase with no bytes
    return;
  }
  if (*host_fill) {  // last written by cp.async: order that before the bulk copies' writes
    fence_proxy_async_smem();
    *host_fill = 0u;
  }
  const int inp = d.down ? I : H;
  const uint32_t rb = inp * d.bits / 8, sp = inp / 32;
  const int rows = d.down ? 64 : 32;
  mbar_expect_tx(bar, rows * (rb + 2 * sp));
  const uint8_t *c = d.rec + d.q.w, *sc = d.rec + d.q.s, *bi = d.rec + d.q.b;
  uint8_t *sdst = st + rows * rb;
  if (d.down) {
    bulk_g2s(st, c + (size_t)d.row0 * rb, 64 * rb, bar);
    bulk_g2s(sdst, sc + (size_t)d.row0 * sp, 64 * sp, bar);
    bulk_g2s(sdst + 64 * sp, bi + (size_t)d.row0 * sp, 64 * sp, bar);
  } else {
    bulk_g2s(st, c + (size_t)d.row0 * rb, 16 * rb, bar);
    bulk_g2s(st + 16 * rb, c + (size_t)(I + d.row0) * rb, 16 * rb, bar);
    bulk_g2s(sdst, sc + (size_t)d.row0 * sp, 16 * sp, bar);
    bulk_g2s(sdst + 16 * sp, sc + (size_t)(I + d.row0) * sp, 16 * sp, bar);
    bulk_g2s(sdst + 32 * sp, bi + (size_t)d.row0 * sp, 16 * sp, bar);
    bulk_g2s(sdst + 48 * sp, bi + (size_t)(I + d.row0) * sp, 16 * sp, bar);
  }
}

// Top-k and softmax of row b by warp b (b < nb), from lg[b][E1 stride].
__device__ __forceinline__ void topk_rows(const float *lg, int E1, int E, int K, int nb, int *sidx, float *sw) {
  const int warp = threadIdx.x >> 5;
  if (warp >= nb) return;
  if (E <= 128)
    topk_warp<4>(lg + warp * E1, E, K, sidx + warp * 32, sw + warp * 32);
  else if (E <= 256)
    topk_warp<8>(lg + warp * E1, E, K, sidx + warp * 32, sw + warp * 32);
  else if (E <= 512)
    topk_warp<16>(lg + warp * E1, E, K, sidx + warp * 32, sw + warp * 32);
  else
    topk_warp<32>(lg + warp * E1, E, K, sidx + warp * 32, sw + warp * 32);
}

// Lookahead, step 1 (every thread of the CTA): this CTA's rows of layer
// l + 1's router on layer l's staged input xf, published to the lookahead
// buffer with tag l + 2.  red: scratch of at least 256 floats.
__device__ __noinline__ void lookahead_rows(const FwdParams &P, int l, const float *xf, float *red) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, cta = blockIdx.x, H = P.H, E = P.E, nb = P.nb, nch = H / 256;
  const LayerP &Ln = P.L[l + 1];
  const int q0 = fdiv_mul(cta, E, G), q1 = fdiv_mul(cta + 1, E, G);
  const int nq = (q1 - q0) * nch;
  __syncthreads();  // red is free again (the caller's sums are published)
  uint4 pv[4];
#pragma unroll
  for (int k = 0; k < 4; k++) {
    const int it = warp + k * NW;
    if (it < nq) pv[k] = ldg_stream4(Ln.router + (size_t)(q0 + it / nch) * H + (it % nch) * 256 + lane * 8);
  }
#pragma unroll
  for (int k = 0; k < 4; k++) {
    const int it = warp + k * NW;
    if (it < nq) {
      const int ch = it % nch;
      const float wf[8] = {bf16lo(pv[k].x), bf16hi(pv[k].x), bf16lo(pv[k].y), bf16hi(pv[k].y),
                           bf16lo(pv[k].z), bf16hi(pv[k].z), bf16lo(pv[k].w), bf16hi(pv[k].w)};
      for (int b = 0; b < nb; b++) {
        const float4 *xp = reinterpret_cast<const float4 *>(xf + b * H + ch * 256 + lane * 8);
        const float4 x0 = xp[0], x1 = xp[1];
        float acc = wf[0] * x0.x + wf[1] * x0.y + wf[2] * x0.z + wf[3] * x0.w + wf[4] * x1.x + wf[5] * x1.y +
                    wf[6] * x1.z + wf[7] * x1.w;
        acc = warp_sum(acc);
        if (lane == 0) red[it * 4 + b] = acc;
      }
    }
  }
  __syncthreads();
  for (int j = tid; j < (q1 - q0) * nb; j += NT) {
    const int r = j / nb, b = j % nb;
    float sum = 0.f;
    for (int ch = 0; ch < nch; ch++) sum += red[(r * nch + ch) * 4 + b];
    st_relaxed_u64(P.lgp + ((size_t)((l + 1) & 1) * kMaxGrid + cta) * kLogitWords + j,
                   ((unsigned long long)(l + 2) << 32) | __float_as_uint(sum));
  }
}

// Lookahead, step 2 (warp 0): the predicted experts' records (device memory
// on this GPU only) laid end to end; this CTA prefetches its 1/G share of
// those bytes into L2.  Lane j takes predicted experts j and j + 32.
__device__ __noinline__ void lookahead_prefetch(const LayerP &Ln, const int *puni, int Up) {
  const int lane = threadIdx.x & 31, G = gridDim.x, cta = blockIdx.x;
  uint64_t spn[2] = {0, 0};
  const uint8_t *base[2] = {nullptr, nullptr};
#pragma unroll
  for (int h = 0; h < 2; h++) {
    const int j = lane + 32 * h;
    if (j < Up) {
      const int e = puni[j];
      const uint64_t a = Ln.eaddr[e];
      const int t = Ln.etier ? Ln.etier[e] : 0;
      const int b = Ln.ebits ? Ln.ebits[e] : 4;
      if (a != 0 && t == 0 && b >= 2 && b <= 4) {
        spn[h] = Ln.ebits ? Ln.span_w[4 - b] : Ln.span;
        base[h] = reinterpret_cast<const uint8_t *>(a);
      }
    }
  }
  uint64_t inc[2] = {spn[0], spn[1]};
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int h = 0; h < 2; h++) {
      const uint64_t v = __shfl_up_sync(FULL, inc[h], o);
      if (lane >= o) inc[h] += v;
    }
  }
  const uint64_t tot0 = __shfl_sync(FULL, inc[0], 31), tot = tot0 + __shfl_sync(FULL, inc[1], 31);
  const uint64_t lo = (tot * (uint64_t)cta / G) & ~255ull;
  const uint64_t hi = cta + 1 == G ? tot : (tot * (uint64_t)(cta + 1) / G) & ~255ull;
#pragma unroll
  for (int h = 0; h < 2; h++) {
    const uint64_t st = (h == 0 ? 0 : tot0) + inc[h] - spn[h];
    const uint64_t a = st > lo ? st : lo, z = st + spn[h] < hi ? st + spn[h] : hi;
    for (uint64_t o = a; o < z; o += 65536) {
      const uint64_t n = z - o < 65536 ? z - o : 65536;
      prefetch_l2(base[h] + (o - st), (uint32_t)n);
    }
  }
}

// Lookahead, step 2 (every thread of the CTA, once its units are done):
// the predicted logits into lg, top-k per row, their union, the predicted
// ids to the next layer's lookahead output (CTA 0), and this CTA's share of
// the prefetch.  red (free again by now) holds the union and its scratch.
__device__ __noinline__ void lookahead_step(const FwdParams &P, int l, float *lg, int E1, int *sidx, float *sw,
                                            int *posof, float *red) {
  const int tid = threadIdx.x, warp = tid >> 5, nb = P.nb, K = P.K, E = P.E;
  const LayerP &Ln = P.L[l + 1];
  int *puni = reinterpret_cast<int *>(red + 1024);
  volatile int *pnu = puni + 64;
  float *pwm = red + 2048;
  const bool got = __syncthreads_and(
      read_tagged(P, P.lgp + (size_t)((l + 1) & 1) * kMaxGrid * kLogitWords, (unsigned)l + 2u, E, E1, lg, true));
  if (got) {
    topk_rows(lg, E1, E, K, nb, sidx, sw);
    __syncthreads();
    if (warp == 0) union_warp(sidx, sw, nb, K, puni, pwm, posof, reinterpret_cast<int *>(red), pnu);
    __syncthreads();
    if (blockIdx.x == 0 && Ln.la_idx)
      for (int j = tid; j < nb * K; j += NT) Ln.la_idx[j] = (uint32_t)sidx[(j / K) * 32 + j % K];
    if (warp == 0) lookahead_prefetch(Ln, puni, *pnu);
  } else if (blockIdx.x == 0 && Ln.la_idx) {
    for (int j = tid; j < nb * K; j += NT) Ln.la_idx[j] = 0xffffffffu;
  }
  __syncthreads();  // lg, sidx, sw, red are the next layer's again
}

// Whether layer l predicts layer l + 1 (its flag; a call that computes
// experts; at most four router items per warp and one CTA's words in a row
// of the lookahead buffer).
__device__ __forceinline__ bool lookahead_on(const FwdParams &P, int l, int G) {
  const int rows = (P.E + G - 1) / G;
  return l + 1 < P.nl && (P.L[l + 1].flags & kLookahead) && !P.route_only && rows * (P.H / 256) <= 4 * NW &&
         rows * P.nb <= kLogitWords;
}

// ------------------------------------------------------------ the kernel

// LA: some layer of the call has the lookahead flag (the instance without
// it carries none of the lookahead's code).
template <int BITS, bool LA>
__global__ void __launch_bounds__(NT, 1) decode_kernel(const __grid_constant__ FwdParams P) {
  // launched as a programmatic dependent of zero_call: wait for the zeroed
  // counters and status before anything else
  asm volatile("griddepcontrol.wait;" ::: "memory");
  extern __shared__ __align__(128) unsigned char sm[];
  const int H = P.H, E = P.E, K = P.K, I = P.I, nb = P.nb;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  const int nblkH = H / 128, nblkI = I / 128;
  const int E1 = (E + 1 + 3) & ~3;
  const int ng = H / 64;
  const int S = P.stages;
  // codec order of the routed activation fragments: BITS's own, or the
  // 4-bit order that every width can read when the union mixes widths
  constexpr int AB = BITS == 0 ? 4 : BITS;

  uint8_t *stages = sm;                                                  // [S][stage_bytes]
  float *xf = reinterpret_cast<float *>(sm + (size_t)S * P.stage_bytes);  // [nb][H]
  uint2 *xa = reinterpret_cast<uint2 *>(xf + nb * H);                    // [nblkH][8][32] routed codec order
  uint2 *xa4 = AB == 4 ? xa : xa + nblkH * 256;                          // shared (4-bit) order
  float *xs = reinterpret_cast<float *>(xa4 + nblkH * 256);              // [4][H/64] group sums of x
  float *cs = xs + 4 * ng;                                               // [4][H/64] offset sums, routed order
  float *cs4 = cs + 4 * ng;                                              // [4][H/64] offset sums, 4-bit order
  float *lg = cs4 + 4 * ng;                                              // [4][E1]
  float *red = lg + 4 * E1;                                              // [2][2048]: one per unit group
  int *sidx = reinterpret_cast<int *>(red + 2 * 2048);                   // [4][32]
  float *sw = reinterpret_cast<float *>(sidx + 128);                     // [4][32]
  int *uni = reinterpret_cast<int *>(sw + 128);                          // [64]
  float *wm = reinterpret_cast<float *>(uni + 64);                       // [4][64]
  float *gam = wm + 256;                                                 // [4]
  volatile int *sflag = reinterpret_cast<volatile int *>(gam + 4);       // [12]
  uint64_t *bars = reinterpret_cast<uint64_t *>(gam + 16);               // [kMaxStages]
  const uint8_t **rect = reinterpret_cast<const uint8_t **>(bars + kMaxStages);  // [64] slot -> record
  // per unit group: staged h fragments [I/128 * 256], their sums [4][I/64], offset sums [4][I/64]
  uint2 *hsm = reinterpret_cast<uint2 *>(rect + 64);
  const int hsz = nblkI * 256 * 2 + 2 * 64;  // 32-bit words per group
  uint64_t *eaddr_s = reinterpret_cast<uint64_t *>(reinterpret_cast<uint32_t *>(hsm) + 2 * hsz);  // [E]
  unsigned *stg_unit = reinterpret_cast<unsigned *>(eaddr_s + ((E + 1) & ~1));  // [S] last unit issued per stage
  unsigned *stg_host = stg_unit + kMaxStages;                                    // [S] stage last filled by cp.async
  int *posof = reinterpret_cast<int *>(stg_host + kMaxStages);                   // [E] union scratch, INT_MAX between uses
  int *sbits = posof + E;                                                        // [64] slot -> code width (mixed)
  int *stier = sbits + 64;                                                       // [64] slot -> record in host memory
  volatile int *absent = stier + 64;                                             // [4] [0]: some record of the layer not on this GPU
  uint8_t *eb_s = reinterpret_cast<uint8_t *>(stier + 68);                       // [E] expert -> code width (mixed)
  uint8_t *et_s = eb_s + ((E + 15) & ~15);                                       // [E] expert -> record in host memory

  if (tid == 0) {
    for (int s = 0; s < S; s++) mbar_init(&bars[s], 1), stg_unit[s] = 0xffffffffu, stg_host[s] = 0u;
    absent[0] = 0;
    fence_mbar_init();
    sflag[9] = 0;
  }
  // activation registers and sums: rows b >= nb stay zero for the whole call
  for (uint32_t *z = reinterpret_cast<uint32_t *>(xa) + tid; z < reinterpret_cast<uint32_t *>(cs4 + 4 * ng); z += NT)
    *z = 0u;
  for (int e = tid; e < E; e += NT) posof[e] = 0x7fffffff;
  __syncthreads();
  // warp lane 0 of an issuing warp: unit q of the layer into its ring stage
  auto issue_at = [&](const UnitDesc &d, unsigned u) {
    issue_unit(d, H, I, stages + (size_t)(u % S) * P.stage_bytes, &bars[u % S], P.status, &stg_host[u % S]);
    if (lane == 0) stg_unit[u % S] = u;
  };

  unsigned qbase = 0;  // units requested so far in this call (ring position)
  for (int l = 0; l < P.nl; l++) {
#define MOE_STAMP(k)                                                                             \
  if (P.trace && tid == 0 && cta < kTraceCtas)                                                   \
    P.trace[((size_t)l * kTraceCtas + cta) * kTracePhases + (k)] = globaltimer();
    MOE_STAMP(0)
    if (l == 0 && tid == 0) sflag[8] = 0;
    const LayerP &L = P.L[l];
    if (LA && l == 0 && cta == 0 && L.la_idx && (L.flags & kLookahead))  // no layer predicts the first one
      for (int j = tid; j < nb * K; j += NT) L.la_idx[j] = 0xffffffffu;
    unsigned *cnt = P.cnt + (size_t)l * kCntPerLayer;
    const bool hs = L.sgate != nullptr;
    const float *src = l == 0 ? P.x : P.xbuf + (size_t)l * nb * H;
    float *dst = l == P.nl - 1 ? P.out : P.xbuf + (size_t)(l + 1) * nb * H;

    Sched s;
    s.hsi = hs ? 1 : 0;
    s.ups = I / 16;
    s.nrt = H / 64;
    s.nA = hs && !P.route_only ? rr_count(cta, s.ups, G) : 0;
    s.nGU = s.nA, s.nD = 0;  // until routing is known
    s.U = 0;
    int issued = 0;
    if (warp == kProducerWarp) {
      for (; issued < s.nA && issued < S; issued++)
        issue_at(get_unit<BITS>(issued, s, L, rect, sbits, stier), qbase + issued);
    }
    issued = s.nA < S ? s.nA : S;

    // ---- R: input, norm, fragments, router rows
    // Loads that need no input go first, so they overlap the wait for the
    // previous layer: this CTA's router rows (every load of a warp in
    // flight at once, <= 4 items per warp) and the expert addresses.
    const int R = E + s.hsi;
    const int rr0 = fdiv_mul(cta, R, G), rr1 = fdiv_mul(cta + 1, R, G);
    const int nch = H / 256;
    const int nitem = (rr1 - rr0) * nch;
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
    for (int e = tid; e < E; e += NT) {
      const uint64_t a = L.eaddr[e];
      eaddr_s[e] = a;
      if (a == 0ull) absent[0] = 1;  // (cleared at the end of every layer)
    }
    if (BITS == 0)
      for (int e = tid; e < E; e += NT) eb_s[e] = L.ebits[e];
    if (L.etier)
      for (int e = tid; e < E; e += NT) et_s[e] = L.etier[e];
    if (l > 0 && !cta_wait(P.cnt + (size_t)(l - 1) * kCntPerLayer + kCntRows, (unsigned)(H / 64), P, sflag)) {
      drain_ring(bars, qbase, qbase + issued, S, P);
      return;
    }
    MOE_STAMP(1)
    const int n4 = nb * H / 4, h4 = H / 4;
    const bool norm = (L.flags & kPrenorm) != 0;
    {
      // the raw input to shared memory in one round trip (each thread up to
      // 4 float4 of the nb rows); with the unit RMSNorm, the rows' sums of
      // squares as warp partials (red[1024 + warp * 4 + b])
      const float4 *src4 = reinterpret_cast<const float4 *>(src);
      float4 *xf4 = reinterpret_cast<float4 *>(xf);
      float4 v[4];
#pragma unroll
      for (int k = 0; k < 4; k++) {
        const int i = tid + k * NT;
        v[k] = i < n4 ? __ldcg(src4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int k = 0; k < 4; k++) {
        const int i = tid + k * NT;
        if (i < n4) xf4[i] = v[k];
      }
      if (norm) {
        float ss[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < 4; k++) {
          const int i = tid + k * NT;
          if (i < n4) ss[i / h4] += v[k].x * v[k].x + v[k].y * v[k].y + v[k].z * v[k].z + v[k].w * v[k].w;
        }
#pragma unroll
        for (int b = 0; b < 4; b++) ss[b] = warp_sum(ss[b]);
        if (lane == 0)
          for (int b = 0; b < 4; b++) red[1024 + warp * 4 + b] = ss[b];
      }
    }
    __syncthreads();
    // this CTA's router rows on the raw input: the norm is one scalar per
    // row, applied to the sums as they are published, so the logits leave
    // before the input's tensor-core fragments are staged
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
          float acc = wf[0] * x0.x + wf[1] * x0.y + wf[2] * x0.z + wf[3] * x0.w + wf[4] * x1.x + wf[5] * x1.y +
                      wf[6] * x1.z + wf[7] * x1.w;
          acc = warp_sum(acc);
          if (lane == 0) red[it * 4 + b] = acc;
        }
      }
    }
    __syncthreads();
    // row scales 1 / sqrt(mean(x^2) + 1e-6), formed by every thread from the
    // warp partials in a fixed order (the same value everywhere)
    float rs[4] = {1.f, 1.f, 1.f, 1.f};
    if (norm) {
#pragma unroll
      for (int b = 0; b < 4; b++) {
        if (b < nb) {
          float t = 0.f;
          for (int w = 0; w < NW; w++) t += red[1024 + w * 4 + b];
          rs[b] = 1.0f / sqrtf(t / (float)H + 1e-6f);
        }
      }
    }
    for (int j = tid; j < (rr1 - rr0) * nb; j += NT) {
      const int r = j / nb, b = j % nb;
      float sum = 0.f;
      for (int ch = 0; ch < nch; ch++) sum += red[(r * nch + ch) * 4 + b];
      sum *= rs[b];
      // value and layer tag in one 64-bit store: no release fence
      if (!(P.withhold && rr0 + r == 0))
        st_relaxed_u64(P.lgw + ((size_t)(l & 1) * kMaxGrid + cta) * kLogitWords + j,
                       ((unsigned long long)(l + 1) << 32) | __float_as_uint(sum));
    }
    MOE_STAMP(3)
    // the normalised input and its fragments, while the other CTAs' logits
    // arrive
    if (norm) {
      float4 *xf4 = reinterpret_cast<float4 *>(xf);
#pragma unroll
      for (int k = 0; k < 4; k++) {
        const int i = tid + k * NT;
        if (i < n4) {
          const float r = rs[i / h4];
          float4 q = xf4[i];
          q.x *= r, q.y *= r, q.z *= r, q.w *= r;
          xf4[i] = q;
        }
      }
    }
    __syncthreads();
    stage_frags<AB>(xf, H, nb, xa, xs, cs);
    if (AB != 4 && hs) stage_frags<4>(xf, H, nb, xa4, nullptr, cs4);
    MOE_STAMP(2)
    // ---- lookahead: this CTA's rows of the next layer's router on this
    // layer's input, published for the prediction of the next layer's
    // experts (rows split over the CTAs as the exact ones are; one pass of
    // at most four items per warp, so long rows or few CTAs go without)
    if (LA && lookahead_on(P, l, G)) lookahead_rows(P, l, xf, red);

    // ---- T: top-k, softmax, union
    // every logit of the layer, each polled until its writer's tag shows
    if (!__syncthreads_and(read_logits(P, l, R, E1, lg))) {
      drain_ring(bars, qbase, qbase + issued, S, P);
      return;
    }
    MOE_STAMP(4)
    MOE_STAMP(8)
    topk_rows(lg, E1, E, K, nb, sidx, sw);
    if (tid < 4) gam[tid] = (hs && tid < nb) ? 1.f / (1.f + expf(-lg[tid * E1 + E])) : 0.f;
    __syncthreads();
    MOE_STAMP(9)
    if (warp == 0) {
      union_warp(sidx, sw, nb, K, uni, wm, posof, reinterpret_cast<int *>(red), sflag + 1);
      if (absent[0] || L.etier || L.cut_w > 0.f) {
        place_union(uni, wm, eaddr_s, L.etier ? et_s : nullptr, L.cut_w, sflag[1], stier + s.hsi, sflag + 2);
        if (lane == 0 && s.hsi) stier[0] = 0;  // the shared expert's record is in device memory
      } else {
        // every record in device memory on this GPU, none cut: the union as it is
        for (int j = lane; j < 64; j += 32) stier[j] = 0;
        if (lane == 0) sflag[2] = sflag[1], sflag[3] = sflag[1];
      }
    }
    __syncthreads();
    MOE_STAMP(10)
    const int Uall = sflag[1];
    s.U = sflag[2];  // the slots this GPU computes
    const int Udev = sflag[3];
    if (tid < s.U) {
      rect[tid + s.hsi] = reinterpret_cast<const uint8_t *>(eaddr_s[uni[tid]]);
      if (BITS == 0) {
        const int b = eb_s[uni[tid]];
        // a width outside {2, 3, 4} is reported; its units then read the
        // fewest bytes (2-bit), which stay inside a record of any width
        if (b < 2 || b > 4) atomicCAS(P.status, 0, kStatusDevice);
        sbits[tid + s.hsi] = b >= 2 && b <= 4 ? b : 2;
      }
    }
    if (cta == 0) {
      if (P.slot_tab)
        for (int j = tid; j < kSlotStride; j += NT) {
          uint64_t v = j < s.U ? eaddr_s[uni[j]] : 0ull;
          if (j == kSlotStride - 2) v = (uint64_t)Udev;
          if (j == kSlotStride - 1) v = (uint64_t)Uall;
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
    if (P.route_only) {
      if (tid == 0) absent[0] = 0;
      __syncthreads();  // eaddr_s is rewritten at the top of the next layer
      continue;
    }

    // ---- schedule of this CTA's units for the layer
    __syncthreads();
    s.nslots = s.U + s.hsi;
    s.nGU = rr_count(cta, s.nslots * s.ups, G);
    s.nD = rr_count(cta, s.nslots * s.nrt, G);
    const int n = s.n();
    if (warp == kProducerWarp) {
      for (int q = issued; q < n && q < S; q++) issue_at(get_unit<BITS>(q, s, L, rect, sbits, stier), qbase + q);
    }
    issued = n < S ? n : S;
    if (s.nslots == 0) {
      // nothing of this layer is resident here (an expert-parallel shard
      // whose experts no row chose, without the shared expert): the output
      // is the residual, or zero; CTA c writes 64-row ranges c, c + G, ...
      for (int rt = cta; rt < ng; rt += G) {
        for (int j = tid; j < 64 * nb; j += NT) {
          const int r = j & 63, b = j >> 6;
          const size_t o = (size_t)b * H + rt * 64 + r;
          dst[o] = (L.flags & kResidual) ? __ldcg(src + o) : 0.f;
        }
        __syncthreads();
        if (tid == 0) red_release_add(cnt + kCntRows, 1u);
      }
    }

    // ---- G + D: the unit loop, each group taking the next free unit
    MOE_STAMP(5)
    {
      const int grp = warp / GW, gw = warp % GW, gt = tid % GT;
      float *gred = red + grp * 2048;
      uint2 *ghsm = reinterpret_cast<uint2 *>(reinterpret_cast<uint32_t *>(hsm) + grp * hsz);
      float *ghxs = reinterpret_cast<float *>(ghsm + nblkI * 256), *ghcs = ghxs + 64;
      volatile int *gflag = sflag + 4 + 2 * grp;  // [0]: wait outcome, [1]: last-unit ticket
      int cur = -1;
      bool alive = true;
      // stamp k from whichever group runs the unit
#define MOE_GSTAMP(k)                                                                            \
  if (P.trace && gt == 0 && cta < kTraceCtas)                                                    \
    P.trace[((size_t)l * kTraceCtas + cta) * kTracePhases + (k)] = globaltimer();
      // the groups take the layer's units in order, each the next free one
      // (sflag[9]: next unit; sflag[10 + g]: group g's pick), so neither
      // group idles while the other still has several units
      for (;;) {
        if (gt == 0) sflag[10 + grp] = atomicAdd(const_cast<int *>(sflag + 9), 1);
        grp_sync(grp);
        const int q = sflag[10 + grp];
        if (q >= n || !alive) break;
        if (q == s.nGU) {
          MOE_GSTAMP(6)
          if (gt == 0 && l + 1 < P.nl) {
            // the next layer's router rows of this CTA, toward L2 while the down units run
            const LayerP &Ln = P.L[l + 1];
            const int re = rr1 < E ? rr1 : E;
            if (re > rr0) prefetch_l2(Ln.router + (size_t)rr0 * H, (uint32_t)((re - rr0) * H * 2));
            if (rr1 > E && Ln.sgate) prefetch_l2(Ln.sgate, (uint32_t)(H * 2));
          }
        }
        const UnitDesc d = get_unit<BITS>(q, s, L, rect, sbits, stier);
        const unsigned u = qbase + q;
        const uint8_t *st = stages + (size_t)(u % S) * P.stage_bytes;
        const bool shared = s.hsi && d.slot == 0;
        if (d.down && d.slot != cur) {
          // h of this slot complete?  then stage its fragments and group sums
          if (!grp_wait(cnt + kCntGu + d.slot * kCntPad, (unsigned)s.ups, P, gflag, grp, gt)) {
            alive = false;
            break;
          }
          cur = d.slot;
          const uint2 *hf = reinterpret_cast<const uint2 *>(P.hfrag) + (size_t)d.slot * nblkI * 256;
          if (shared || AB == 4)
            stage_h<4>(hf, I, nb, ghsm, ghxs, ghcs, grp, gt);
          else
            stage_h<AB>(hf, I, nb, ghsm, ghxs, ghcs, grp, gt);
        }
        if (!grp_and(grp, stage_wait(&bars[u % S], (u / S) & 1u, P))) {
          alive = false;
          break;
        }
        if (q == 0) MOE_STAMP(11)
        const bool ok = d.rec != nullptr && ((uintptr_t)d.rec & 15u) == 0;
        if (ok) {
          const int rows = d.down ? 64 : 32, inp = d.down ? I : H;
          const uint32_t *sw = reinterpret_cast<const uint32_t *>(st + rows * code_pitch(inp * d.bits / 8, d.bits));
          const float *csx = shared && AB != 4 ? cs4 : cs;
          const uint2 *xbx = shared ? xa4 : xa;
          // the unit's codec: 4-bit for the shared expert, BITS's own, or
          // (mixed widths) the slot's width read in the 4-bit pair order
          const int cb = shared ? 4 : (BITS == 0 ? d.bits : BITS);
          if (!d.down) {
            if (nb <= 2) {
              if (cb == 4) gate_up_compute<4, 1>(st, sw, H, xbx, xs, csx, nb, gred, gw, GW);
              else if (BITS == 0 && cb == 3) gate_up_compute<3, 1, true>(st, sw, H, xbx, xs, csx, nb, gred, gw, GW);
              else if (BITS == 0) gate_up_compute<2, 1, true>(st, sw, H, xbx, xs, csx, nb, gred, gw, GW);
              else gate_up_compute<AB, 1>(st, sw, H, xbx, xs, csx, nb, gred, gw, GW);
            } else {
              if (cb == 4) gate_up_compute<4, 2>(st, sw, H, xbx, xs, csx, nb, gred, gw, GW);
              else if (BITS == 0 && cb == 3) gate_up_compute<3, 2, true>(st, sw, H, xbx, xs, csx, nb, gred, gw, GW);
              else if (BITS == 0) gate_up_compute<2, 2, true>(st, sw, H, xbx, xs, csx, nb, gred, gw, GW);
              else gate_up_compute<AB, 2>(st, sw, H, xbx, xs, csx, nb, gred, gw, GW);
            }
          } else {
            if (nb <= 2) {
              if (cb == 4) down_compute<4, 1>(st, sw, I, ghsm, ghxs, ghcs, nb, gred, gw, GW);
              else if (BITS == 0 && cb == 3) down_compute<3, 1, true>(st, sw, I, ghsm, ghxs, ghcs, nb, gred, gw, GW);
              else if (BITS == 0) down_compute<2, 1, true>(st, sw, I, ghsm, ghxs, ghcs, nb, gred, gw, GW);
              else down_compute<AB, 1>(st, sw, I, ghsm, ghxs, ghcs, nb, gred, gw, GW);
            } else {
              if (cb == 4) down_compute<4, 2>(st, sw, I, ghsm, ghxs, ghcs, nb, gred, gw, GW);
              else if (BITS == 0 && cb == 3) down_compute<3, 2, true>(st, sw, I, ghsm, ghxs, ghcs, nb, gred, gw, GW);
              else if (BITS == 0) down_compute<2, 2, true>(st, sw, I, ghsm, ghxs, ghcs, nb, gred, gw, GW);
              else down_compute<AB, 2>(st, sw, I, ghsm, ghxs, ghcs, nb, gred, gw, GW);
            }
          }
        }
        grp_sync(grp);
        if (q == 0) MOE_STAMP(12)
        // the stage is free: request the unit S places ahead into it
        if (gw == kProducerWarp && q + S < n) issue_at(get_unit<BITS>(q + S, s, L, rect, sbits, stier), u + S);
        if (!d.down) {
          // h = silu(gate) * up for 16 rows x nb, scattered as bf16 hi/lo A
          // fragments in the pair order of this slot's down codec; thread
          // (i, b) sums its gate and up rows over the blocks in block order
          if (gt < 16 * nb) {
            const int i = gt & 15, b = gt >> 4;
            float gsum = 0.f, usum = 0.f;
            for (int kb = 0; kb < nblkH; kb++) {
              gsum += gred[(kb * 2) * 64 + i * 4 + b];
              usum += gred[(kb * 2 + 1) * 64 + i * 4 + b];
            }
            const float h = ok ? gsum / (1.f + expf(-gsum)) * usum : 0.f;
            const int pos = d.row0 + i;
            const int blk = pos >> 7, c = pos & 127, tq = c >> 5, cc = c & 31;
            int pi = 0, el = 0, sh = 0;
#pragma unroll
            for (int p = 0; p < 16; p++) {
              const bool c4 = shared || AB == 4;
              const int lo = c4 ? Codec<4>::lo(p) : Codec<AB>::lo(p);
              const int hi = c4 ? Codec<4>::hi(p) : Codec<AB>::hi(p);
              if (lo == cc) pi = p, el = 0, sh = c4 ? Codec<4>::slo(p) : Codec<AB>::slo(p);
              if (hi == cc) pi = p, el = 1, sh = c4 ? Codec<4>::shi(p) : Codec<AB>::shi(p);
            }
            const float hv = h * __uint_as_float((uint32_t)(127 - sh) << 23);  // h * 2^-sh, exact
            const uint32_t hi = f2bf(hv), lo = f2bf(hv - __uint_as_float(hi << 16));
            uint16_t *hb = P.hfrag + (size_t)d.slot * nblkI * 256 * 4;
            const int m = pi >> 1, reg = pi & 1;
            hb[frag_index(blk, b >> 1, m, tq, 0, b & 1) * 4 + reg * 2 + el] = (uint16_t)hi;
            hb[frag_index(blk, b >> 1, m, tq, 1, b & 1) * 4 + reg * 2 + el] = (uint16_t)lo;
          }
          grp_signal(cnt + kCntGu + d.slot * kCntPad, 1u, grp, gt);
          if (q == 0) MOE_STAMP(13)
          if (q == s.nGU - 1) MOE_GSTAMP(14)
        } else {
          const int rt = d.row0 / 64;
          for (int j = gt; j < 64 * nb; j += GT) {
            const int r = j & 63, b = j >> 6;
            float y = 0.f;
            if (ok)
              for (int kb = 0; kb < nblkI; kb++) y += gred[(kb * 4 + (r >> 4)) * 64 + (r & 15) * 4 + b];
            const float mb = shared ? gam[b] : wm[b * 64 + d.slot - s.hsi];
            P.ypart[((size_t)d.slot * nb + b) * H + d.row0 + r] = mb * y;
          }
          grp_sync(grp);
          if (gt == 0) gflag[1] = atom_acq_rel_add(cnt + kCntDn + rt * kCntPad, 1u) == (unsigned)(s.nslots - 1);
          grp_sync(grp);
          if (gflag[1]) {
            // last unit of this 64-row range: sum the slots in a fixed order
            const int tpo = nb == 1 ? 8 : (nb == 2 ? 4 : 2);
            for (int j = gt; j < 64 * nb * tpo; j += GT) {
              const int o = j / tpo, part = j % tpo;
              const int r = o & 63, b = o >> 6;
              const float *yp = P.ypart + (size_t)b * H + d.row0 + r;
              float acc = 0.f;
#pragma unroll 4
              for (int sl = part; sl < s.nslots; sl += tpo) acc += __ldcg(yp + (size_t)sl * nb * H);
              for (int off = tpo >> 1; off; off >>= 1) acc += __shfl_down_sync(FULL, acc, off, tpo);
              if (part == 0) {
                if (L.flags & kResidual) acc += __ldcg(src + (size_t)b * H + d.row0 + r);
                dst[(size_t)b * H + d.row0 + r] = acc;
              }
            }
            grp_signal(cnt + kCntRows, 1u, grp, gt);
          }
          grp_sync(grp);
          if (q == s.nGU) MOE_GSTAMP(15)
        }
      }
      if (!alive) sflag[8] = 1;
#undef MOE_GSTAMP
    }
    __syncthreads();  // both groups are done with the layer's units
    if (sflag[8]) {
      drain_stages(bars, stg_unit, S, P);
      return;
    }
    // ---- lookahead: predict the next layer's experts and prefetch this
    // CTA's share of their records into L2, now that this CTA's units are
    // done: the prefetches overlap the wait for the next layer's input and
    // its routing
    if (LA && lookahead_on(P, l, G)) lookahead_step(P, l, lg, E1, sidx, sw, posof, red);
    if (tid == 0) sflag[9] = 0, absent[0] = 0;  // the next layer's unit counter and absent flag
    qbase += (unsigned)n;
    MOE_STAMP(7)
#undef MOE_STAMP
  }
}

}  // namespace

static int fixed_smem(int H, int E, int I, int nb, int bits) {
  const int nblkH = H / 128;
  const int E1 = (E + 1 + 3) & ~3;
  int b = 0;
  b += nb * H * 4;                                 // xf
  b += nblkH * 256 * 8 * (bits == 4 || bits == 0 ? 1 : 2);  // xa (+ xa4; one 4-bit order when widths mix)
  b += 3 * 4 * (H / 64) * 4;                       // xs, cs, cs4
  b += 4 * E1 * 4;                                 // lg
  b += 2 * 2048 * 4;                               // red, one per unit group
  b += (128 + 128 + 64 + 256 + 16) * 4;            // sidx sw uni wm gam+flags
  b += kMaxStages * 8;                             // barriers
  b += 64 * 8;                                     // slot -> record table
  b += 2 * ((I / 128) * 256 * 8 + 2 * 64 * 4);     // staged h fragments and sums, one per unit group
  b += ((E + 1) & ~1) * 8;                         // expert addresses
  b += 2 * kMaxStages * 4;                         // last unit issued per stage, stage last filled by cp.async
  b += E * 4;                                      // union scratch
  b += 2 * 64 * 4 + 16 + 2 * ((E + 15) & ~15);     // slot widths and tiers, layer flags, expert widths and tiers
  return b;
}

static int stage_bytes(int H, int I) {
  // the 4-bit tiles are the largest (the shared expert is always 4-bit)
  const int gu = 32 * code_pitch(H * 4 / 8, 4) + 64 * (H / 32);
  const int dn = 64 * code_pitch(I * 4 / 8, 4) + 128 * (I / 32);
  const int m = gu > dn ? gu : dn;
  return (m + 127) & ~127;
}

template <int BITS, bool LA>
static int occupancy_t(int smem) {
  int n = 0;
  if (cudaFuncSetAttribute(decode_kernel<BITS, LA>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<BITS, LA>, NT, smem) != cudaSuccess) return 0;
  return n;
}

template <bool LA>
static int occupancy_b(int bits, int smem) {
  return bits == 4   ? occupancy_t<4, LA>(smem)
         : bits == 3 ? occupancy_t<3, LA>(smem)
         : bits == 2 ? occupancy_t<2, LA>(smem)
                     : occupancy_t<0, LA>(smem);
}

int decode_plan(int device, FwdParams &p, int *grid, int *smem_bytes) {
  int sms = 0, optin = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess) return -1;
  const int fixed = fixed_smem(p.H, p.E, p.I, p.nb, p.bits);
  const int sb = stage_bytes(p.H, p.I);
  int S = (optin - fixed) / sb;
  if (S > kMaxStages) S = kMaxStages;
  if (S < 1) return -1;
  p.stages = S;
  p.stage_bytes = sb;
  const int smem = fixed + S * sb;
  const int occ = p.lookahead ? occupancy_b<true>(p.bits, smem) : occupancy_b<false>(p.bits, smem);
  if (occ < 1) return -1;
  const int G = sms < kMaxGrid ? sms : kMaxGrid;
  // every CTA's router rows x activation rows fit its logit words
  if ((p.E + 1 + G - 1) / G * p.nb > kLogitWords) return -1;
  *grid = G;
  *smem_bytes = smem;
  return 0;
}

// Start of a call: the counters and logit exchange words (n16 16-byte
// units) and the status word to zero.  The decode kernel that follows may
// launch at once and waits for this one with griddepcontrol.wait.
__global__ void zero_call(uint4 *cnt, size_t n16, int *status) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (size_t)gridDim.x * blockDim.x)
    cnt[i] = make_uint4(0u, 0u, 0u, 0u);
  if (blockIdx.x == 0 && threadIdx.x == 0) *status = 0;
}

template <int BITS, bool LA>
static cudaError_t launch_t(const FwdParams &p, int grid, int smem, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, decode_kernel<BITS, LA>, p);
}

template <bool LA>
static cudaError_t launch_b(const FwdParams &p, int grid, int smem, cudaStream_t st) {
  switch (p.bits) {
    case 4: return launch_t<4, LA>(p, grid, smem, st);
    case 3: return launch_t<3, LA>(p, grid, smem, st);
    case 2: return launch_t<2, LA>(p, grid, smem, st);
    case 0: return launch_t<0, LA>(p, grid, smem, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode(const FwdParams &p, int grid, int smem, cudaStream_t st, size_t zero_bytes) {
  const size_t n16 = zero_bytes / 16, blocks = (n16 + 255) / 256;
  zero_call<<<(int)(blocks < 1 ? 1 : blocks > 1024 ? 1024 : blocks), 256, 0, st>>>(reinterpret_cast<uint4 *>(p.cnt), n16,
                                                                                   p.status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return p.lookahead ? launch_b<true>(p, grid, smem, st) : launch_b<false>(p, grid, smem, st);
}

}  // namespace moe
