// decode.cuh -- parameters of the persistent decode / verify kernel (nb <= 4 rows).
#pragma once

#include <cstdint>

#include "common.cuh"

namespace moe {

struct QOff {
  uint32_t w, s, b;  // byte offsets inside a record
};

struct LayerP {
  const uint16_t *router;  // bf16 [E][H]
  const uint16_t *sgate;   // bf16 [H] or nullptr
  const uint8_t *srec;     // shared expert record (4-bit) or nullptr
  const uint64_t *eaddr;   // [E] record base addresses
  QOff gu, dn, sgu, sdn;
  uint32_t flags;
  const uint8_t *ebits;    // [E] code width of each routed record (kernel instance 0, mixed widths)
  QOff guw[3], dnw[3];     // mixed widths: offsets in a record of width 4, 3, 2 (index 4 - width)
  const uint8_t *etier;    // [E] 0: record in device memory, 1: in host memory; nullptr: all in device memory
  float cut_w;             // host-tier experts below this weight in every row are cut (0: none)
  uint32_t span, span_w[3];  // bytes from a record's base to the end of its last tensor (uniform; per width)
  uint32_t *la_idx;        // [nb][K] this layer's experts as predicted one layer early, or nullptr
};

// Per-layer counters in the workspace (uint32 each), every counter on a
// 128-byte line of its own: a line that many SMs poll while others update
// it makes the updates microseconds late.
constexpr int kCntPad = 32;                              // words per counter line
constexpr int kCntRows = 0;                              // 64-row output ranges finalised
constexpr int kCntGu = kCntPad;                          // [64] gate_up units finished per internal slot
constexpr int kCntDn = kCntGu + 64 * kCntPad;            // [H/64 <= 32] down units finished per output range
constexpr int kCntPerLayer = kCntDn + 32 * kCntPad;
constexpr int kMaxGrid = 160;    // CTAs of the decode kernel at most (one per SM)
constexpr int kLogitWords = 32;  // flagged logit words per CTA (two 128-byte lines of one writer)

struct FwdParams {
  int H, E, K, I, nb, nl, bits;  // bits: routed width, or 0 when each record carries its own
  int route_only;
  int withhold;  // failure-detection test: never release the router count
  int lookahead;  // some layer has the lookahead flag (selects the kernel instance that carries it)
  const float *x;
  float *out;
  uint64_t *slot_tab;     // [nl][64] or nullptr
  float *wmap;            // [nl][4][64] or nullptr
  uint32_t *topk_idx;     // [nl][nb][K] or nullptr
  float *topk_w;          // [nl][nb][K] or nullptr
  float *logits_out;      // [nb][E] (route only) or nullptr
  int *status;
  unsigned *cnt;          // [nl][kCntPerLayer]
  unsigned long long *lgp;  // [2][kMaxGrid][kLogitWords] lookahead logits {fp32 bits, layer + 1 predicted}
  unsigned long long *lgw;  // [kMaxGrid][kLogitWords] router logits {fp32 bits, layer + 1}, CTA c's
                            // rows x nb; zeroed per call, reused by every layer
  float *xbuf;            // [nl][nb][H]  input of layer l (l >= 1)
  uint16_t *hfrag;        // [64][I/128][8][32][2][2] bf16 activation fragments of h
  float *ypart;           // [64][nb][H]  per-slot weighted down outputs
  unsigned long long timeout_ns;
  unsigned long long *trace;  // [nl][kTraceCtas][kTracePhases] %globaltimer stamps, or nullptr
  int stages;            // weight-tile ring depth (bulk copies in flight)
  int stage_bytes;       // bytes of one ring stage
  LayerP L[kMaxLayers];
};

constexpr int kMaxStages = 4;
constexpr int kTraceCtas = 1024;
constexpr int kTracePhases = 16;

// Launch helpers (decode.cu)
// Fills p.stages / p.stage_bytes and the grid for this device; returns 0 or -1.
// The grid is one CTA per SM, at most kMaxGrid.
int decode_plan(int device, FwdParams &p, int *grid, int *smem_bytes);
// zero_bytes: the counters and logit exchange words from p.cnt (a multiple of 16), zeroed first with *p.status
cudaError_t launch_decode(const FwdParams &p, int grid, int smem_bytes, cudaStream_t st, size_t zero_bytes);

}  // namespace moe
