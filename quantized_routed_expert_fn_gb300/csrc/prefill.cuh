// prefill.cuh -- parameters of the prefill-chunk path (t rows through one layer).
#pragma once

#include <cuda.h>

#include <cstdint>

#include "decode.cuh"

namespace moe {

struct PfItem {
  int g, mt, n0, nlen;  // group (expert, or E = shared), row tile, first grouped entry, entries
  uint64_t rec;         // the group's record address
};

constexpr int kPfTileN = 160;  // token columns per tensor-core tile
constexpr int kPfChunk = 32;   // tokens per chunk of the stable grouping

struct PfParams {
  // TMA descriptors (bf16, 128B swizzle): router rows [E][H] (box 64 x 128),
  // router operand [2t][H] = x^ hi rows then lo rows (box 64 x 128), the
  // grouped expert operands xc [entries][H] and h [entries][I] (boxes 64 x
  // 128 and 64 x 32)
  CUtensorMap tm_router;
  CUtensorMap tm_xr;
  CUtensorMap tm_xc;
  CUtensorMap tm_xc32;
  CUtensorMap tm_h;
  CUtensorMap tm_h32;
  int H, E, K, I, t;
  int bits;                // routed records' code width (2, 3 or 4); the shared record is 4-bit
  int n_sms;
  uint32_t flags;
  int route_only;          // stop after the grouping
  int withhold;            // failure-detection test: CTA 0 of the gate_up GEMM never completes its first A stage
  const float *x;          // [t][H]
  uint16_t *out;           // bf16 [t][H]
  const uint16_t *router, *sgate;
  const uint8_t *srec;
  const uint64_t *eaddr;
  QOff gu, dn, sgu, sdn;
  uint32_t *topk_out;      // [t][K] or nullptr
  float *topkw_out;        // [t][K] or nullptr
  int *status;
  unsigned long long timeout_ns;
  // workspace
  uint16_t *xr_hi, *xr_lo;  // bf16 [t][H] each, adjacent (xr_lo = xr_hi + t*H): router operand (hi + lo of x^)
  uint16_t *xg;             // bf16 [t][H], x^ rounded, k permuted within 8-blocks: expert operand
  float *gam;               // [t] shared-expert gate
  float *logits;            // [t][E]
  int *tk_idx;              // [t][K]
  float *tk_w;              // [t][K]
  int *chist;               // [E][nch] per-(expert, token chunk) counts, then their places in the list
  int *counts;              // [E] entries per expert
  int *choff;               // [E+2] first chunk (kPfTileN tokens) of each group; choff[G] = chunks
  int *offs;                // [E+2] first grouped entry of each group; offs[G] = total
  int *rows;                // [t*(K+1)] token of each grouped entry
  float *wts;               // [t*(K+1)] its weight
  PfItem *items1, *items2;  // gate_up / down work lists
  int *nitems;              // [2]
  uint16_t *hbuf;           // bf16 [I/64][t*(K+1)][64] (k-panels), k permuted within 8-blocks
  float *Y;                 // [t][H] fp32 accumulator
  uint16_t *xc;             // bf16 [H/64][t*(K+1)][64] (k-panels): xg rows in group order
};

constexpr int kPfStages = 10;  // kernels of one prefill call, in launch order

size_t pf_workspace_bytes(int H, int E, int K, int I, int t);
void pf_carve(PfParams &p, void *work);
// fills the TMA descriptors of p (after pf_carve); 0 on success
int pf_tensor_maps(PfParams &p, const char **why);
// events: nullptr, or kPfStages + 1 events recorded before each kernel and after the last
cudaError_t pf_launch(PfParams &p, cudaStream_t st, cudaEvent_t const *events = nullptr);

}  // namespace moe
