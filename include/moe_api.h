/*
 * moe_api.h -- C ABI of the GB300 routed quantized mixture-of-experts step.
 *
 * The step, for nb consecutive rows of activations x[nb][hidden] (row-major,
 * float32, device memory):
 *   1. router logits L[b][e] = sum_i R[e][i] * x^[b][i], R bf16 [E][hidden]
 *      (x^ = x, or the unit-weight RMSNorm of x with eps 1e-6 when the layer
 *      has MOE_PRENORM);
 *   2. per row the top_k experts by logit (ties to the lower id) and routing
 *      weights = softmax over those k logits;
 *   3. the union of the rows' experts in first-seen order (row-major over the
 *      [nb][top_k] table), published as a slot table of record addresses and a
 *      per-row weight map;
 *   4. each union expert's affine-quantized record evaluated as
 *      gate_up -> silu(gate) * up -> down;
 *   5. out[b] = sum_j wmap[b][j] * y_j[b] + sigmoid(shared_gate . x^[b]) *
 *      y_shared[b]  (+ x[b] when the layer has MOE_RESIDUAL).
 *
 * Sources (qwen4_exp::gpu pages): `Gpu::router_b` (router over nb rows,
 * softmax over experts, top-k) and `Gpu::experts_b` (routed experts of the
 * union published in the slot table, plus the shared expert, summed per row)
 * on the struct Gpu page; the `slot_tab` and `wmap` fields there (per layer
 * SLOT_STRIDE = 64 u64 record addresses, entry 62 the resident count, entry 63
 * the union size; per layer [MAX_NB][64] routing weights); `struct Q`,
 * `Q::at_offset`, `union_of`, `MAX_NB = 4` and `SLOT_STRIDE` on the gpu.rs
 * source page; the load-time checks of load.rs (hidden % 256, expert width a
 * multiple of the 64-code group, top_k * MAX_NB < SLOT_STRIDE, shared width ==
 * expert width, 16-byte aligned code offsets).  The pages do not name the
 * shared gate's activation: sigmoid is the reading taken here.
 *
 * Ownership: the caller allocates every buffer (device memory unless stated);
 * the library allocates nothing and keeps no state between calls.  Calls are
 * asynchronous on the given stream; device-side failures are written to
 * *dev_status (a device int the call zeroes first), readable after a sync.
 * Host-side checks run before any launch; a failing call returns a negative
 * status, launches nothing, and moe_last_error() describes it.
 */
#ifndef MOE_API_H
#define MOE_API_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *moe_stream_t; /* a cudaStream_t; NULL = legacy default stream */

/* One affine-quantized projection (`struct Q`): byte offsets, relative to the
 * record base, of the codes (uint32 words, row-major [out][inp*bits/32], each
 * row one LSB-first bitstream), the scales and the biases (bf16, row-major
 * [out][inp/64]).  Every offset must be 256-byte aligned. */
typedef struct {
  uint64_t w, s, b;
  uint32_t out, inp;
} moe_q;

/* One MoE layer.  A routed record holds gate_up (out = 2*inter: rows
 * 0..inter-1 the gate, inter..2*inter-1 the up projection; inp = hidden) and
 * down (out = hidden, inp = inter).  All layers of one call share hidden,
 * n_experts, top_k, inter and bits. */
typedef struct {
  uint32_t hidden, n_experts, top_k, inter;
  uint32_t bits;  /* routed records: 4, 3 or 2 */
  uint32_t group; /* must be 64 */
  uint32_t flags; /* MOE_RESIDUAL | MOE_PRENORM */
  const uint16_t *router;      /* bf16 [n_experts][hidden] */
  const uint16_t *shared_gate; /* bf16 [hidden]; NULL = no shared expert */
  const void *shared_record;   /* 4-bit record of the shared expert (NULL iff shared_gate is) */
  moe_q sh_gate_up, sh_down;   /* relative to shared_record */
  const uint64_t *expert_addr; /* device array [n_experts] of record base addresses; 0 = the
                                  record is not resident on this GPU (an expert-parallel
                                  shard): the expert is routed as usual but contributes
                                  nothing here (decode; prefill reports MOE_EDEVICE
                                  when a row routes to such an expert) */
  moe_q gate_up, down;         /* relative to each routed record */
  /* Mixed widths (decode only): a union may hold records of different code
   * widths, each keeping its own (the `encode_block` passage of the struct
   * Gpu page: fetched records carry the miss precision, resident ones keep
   * theirs).  NULL: every routed record has `bits` and the offsets above. */
  const uint8_t *expert_bits;   /* device array [n_experts]: 4, 3 or 2 per routed record, or NULL */
  moe_q gate_up_w[3], down_w[3]; /* with expert_bits: the offsets inside a record of width 4, 3
                                    and 2 (index 4 - width); `bits`, gate_up and down unused */
  /* Two-tier records (decode only; the `res` pool and the deadline policy of
   * the struct Gpu page): a routed record lives in device memory or in
   * pinned host memory that the GPU reads directly (its expert_addr is the
   * device pointer of that host memory).  The union is computed device
   * records first, then host ones; slot_tab[62] counts the device ones. */
  const uint8_t *expert_tier; /* device array [n_experts]: 0 device memory, 1 host memory; NULL: all device */
  float cut_weak;             /* host-memory experts whose routing weight is below this in every row of
                                 the call are cut (contribute nothing); 0 = no cut */
  uint32_t *lookahead_idx;    /* device [nb][top_k] or NULL: with MOE_LOOKAHEAD, this layer's experts as
                                 predicted during the previous layer (the lookahead_hit source);
                                 0xffffffff where no prediction was made (first layer of a call) */
} moe_layer;

enum {
  MOE_RESIDUAL = 1, /* out = x + MoE(x^) */
  MOE_PRENORM = 2,  /* x^ = x / sqrt(mean(x^2) + 1e-6) feeds router, gate and experts */
  MOE_LOOKAHEAD = 4, /* decode: while the previous layer of the same call runs, predict this
                        layer's experts from this layer's router applied to the previous
                        layer's input, and prefetch their device-memory records into L2
                        (`lookahead_layer`, struct Gpu page: a one-layer lookahead router);
                        a hint only, results do not change */
  MOE_TEST_WITHHOLD = 0x100 /* failure-detection test only: decode never releases the
                               router's completion, prefill never completes one pipeline
                               stage of its gate_up GEMM; the bounded waits must give up
                               and report MOE_ETIMEOUT */
};

enum moe_status {
  MOE_OK = 0,
  MOE_EINVAL = -1,   /* NULL pointer, bad nb / n_layers, flags, aliasing */
  MOE_ESHAPE = -2,   /* unsupported or inconsistent dimensions */
  MOE_EALIGN = -3,   /* misaligned pointer or offset */
  MOE_ECUDA = -4,    /* a CUDA runtime call failed */
  MOE_ETIMEOUT = -5, /* (device) a bounded wait gave up */
  MOE_EDEVICE = -6,  /* (device) bad data met on the device, e.g. a null record address */
  MOE_ENOSPACE = -7  /* workspace too small */
};

#define MOE_SLOT_STRIDE 64
#define MOE_MAX_NB 4
#define MOE_MAX_LAYERS 64

/* Route one layer: router logits, top-k softmax and the union / slot table.
 *   x        [nb][hidden] float32; nb in 1..4
 *   logits   [nb][n_experts] float32, or NULL
 *   topk_idx [nb][top_k] uint32 (descending logit)
 *   topk_w   [nb][top_k] float32 (sum to 1 per row)
 *   slot_row [64] uint64: record addresses of the union's resident experts
 *            (expert_addr != 0) in first-seen order; [62] = their count,
 *            [63] = the union size (equal when every record is resident)
 *   wmap_row [4][64] float32: row b's weight for slot j of slot_row, else 0
 *   work     device workspace of at least moe_forward_workspace(L, 1, nb) bytes
 * Returns MOE_OK or a negative moe_status. */
int moe_route(const moe_layer *L, const float *x, int nb, float *logits, uint32_t *topk_idx,
              float *topk_w, uint64_t *slot_row, float *wmap_row, void *work, size_t work_bytes,
              int *dev_status, moe_stream_t stream);

/* n_layers stacked MoE layers over nb rows (decode / speculative verify):
 * x_{l+1} = layer_l(x_l), out = x_{n_layers}.  One persistent kernel runs the
 * whole stack; no host round trip between layers.
 *   layers   host array [n_layers] (read during the call only); n_layers in 1..64
 *   x        [nb][hidden] float32; out [nb][hidden] float32, must not overlap x
 *   work     device workspace, at least moe_forward_workspace(layers, n_layers, nb)
 *            bytes, 256-byte aligned; its contents need no initialisation
 *   slot_tab [n_layers][64] uint64, wmap [n_layers][4][64] float32 (see moe_route)
 *   topk_idx [n_layers][nb][top_k] uint32, or NULL
 * Supported shapes: hidden % 256 == 0 and <= 2048, inter % 128 == 0 and <= 1024,
 * n_experts <= 1024, top_k <= 32, top_k * nb < 64, group == 64.
 * Returns MOE_OK or a negative moe_status. */
int moe_forward(const moe_layer *layers, int n_layers, const float *x, int nb, float *out,
                void *work, size_t work_bytes, uint64_t *slot_tab, float *wmap,
                uint32_t *topk_idx, int *dev_status, moe_stream_t stream);

/* moe_forward plus per-phase device timestamps (the `PhaseTimer` / `GpuTiming`
 * GPU timestamps of the struct Gpu page, here %globaltimer nanoseconds).
 *   phase_ns  device array [n_layers][MOE_TRACE_CTAS][MOE_TRACE_PHASES] uint64;
 *             thread 0 of CTA c stamps, for each layer: 0 layer start, 1 layer
 *             input available, 2 input staged, 3 router rows published,
 *             4 all router rows seen, 5 expert units start, 6 first down unit,
 *             7 layer done, 8 logits loaded, 9 top-k done, 10 union done,
 *             11 first unit's tile landed, 12 first unit computed, 13 first
 *             unit published, 14 last gate_up unit published, 15 first down
 *             unit published.  Entries of CTAs beyond the grid, and phases a
 *             CTA skips, are left untouched.
 * Timing costs a few stores per layer; results equal moe_forward's. */
#define MOE_TRACE_CTAS 1024
#define MOE_TRACE_PHASES 16
int moe_forward_traced(const moe_layer *layers, int n_layers, const float *x, int nb, float *out,
                       void *work, size_t work_bytes, uint64_t *slot_tab, float *wmap,
                       uint32_t *topk_idx, int *dev_status, uint64_t *phase_ns, moe_stream_t stream);

/* moe_forward for callers that cannot allocate device memory when they run
 * the step -- e.g. code being captured into a CUDA graph, engines that own
 * all device memory through their own pool, or loops that must not risk the
 * device-wide synchronisation an allocation can cause.  (The pages have no
 * counterpart: their engine sizes all scratch once at load.)
 * Same arguments and results as moe_forward, minus the workspace: the
 * library uses one fixed, process-lifetime device array of
 * MOE_NOALLOC_MAX_WORKSPACE bytes on each GPU that loads it.
 *   - Layers whose moe_forward_workspace exceeds that size are rejected with
 *     MOE_ENOSPACE before anything runs (48 layers of hidden 2048, 128 experts,
 *     inter 768 need about 2.4 MiB at nb 1; the same stack at nb 4 needs 5.0
 *     MiB and is rejected).
 *   - The first call in each CUDA context looks the array's address up once
 *     (cudaGetSymbolAddress with that context current) and keeps it for that
 *     context; make that first call before capturing a stream into a graph.
 *     A cudaDeviceReset ends the context and the array's contents with it:
 *     the next call, in the new context, looks the address up again.
 *   - Every call on a device shares the array, so calls whose executions
 *     overlap on the GPU (different streams, or graph branches) race; order
 *     them on one stream.  Each call clears the parts that must start at zero.
 *   - No allocation or free is made, by the library or any routine it calls. */
#define MOE_NOALLOC_MAX_WORKSPACE (4u << 20)
int moe_forward_noalloc(const moe_layer *layers, int n_layers, const float *x, int nb, float *out,
                        uint64_t *slot_tab, float *wmap, uint32_t *topk_idx, int *dev_status,
                        moe_stream_t stream);

/* Prefill chunk: t rows through ONE layer on the tensor cores (the prefill
 * MoE of the struct Gpu page, `pf_experts`: the shared expert over every row,
 * then the routed experts one at a time -- gather the expert's rows, compute,
 * scatter-add -- with the rows grouped by expert as `ExpertJob` /
 * `prepare_expert_jobs` do).  Per row the routing equals moe_route's (steps
 * 1-2 above); the experts then run as grouped GEMMs with bf16 operands:
 *   x^ is rounded to bf16, every dequantized weight is rounded to bf16
 *   (bf16(scale * code + bias)), h = silu(gate) * up is rounded to bf16, the
 *   products accumulate in fp32, and
 *   out[r] = bf16( sum_j w_j * y_j[r] + sigmoid(shared_gate . x^[r]) *
 *                  y_shared[r]  (+ x[r] when MOE_RESIDUAL) ).
 * The router itself reads x^ at fp32 accuracy (x^ split into two bf16 terms).
 *   L        host pointer to one layer; routed records 4-, 3- or 2-bit (the
 *            shared record is 4-bit); 3-bit records need inter % 128 == 0 so
 *            that their code rows are whole 16-byte pieces
 *   x        [t][hidden] float32, 16-byte aligned; t in 1..1048576
 *   out      [t][hidden] bf16 (uint16 bit patterns); must not overlap x
 *   work     device workspace of at least moe_prefill_workspace(L, t) bytes,
 *            256-byte aligned; its contents need no initialisation
 *   topk_idx [t][top_k] uint32 (descending logit), or NULL
 * Supported shapes: hidden % 256 == 0 (<= 16384), inter % 64 == 0 (<= 16384),
 * n_experts <= 1024, top_k <= 32, group == 64.
 * Returns MOE_OK or a negative moe_status; device-side failures (a null or
 * misaligned record address, a bounded wait that gave up) land in *dev_status. */
int moe_prefill(const moe_layer *L, const float *x, int t, uint16_t *out, void *work, size_t work_bytes,
                uint32_t *topk_idx, int *dev_status, moe_stream_t stream);

/* moe_prefill plus device timing of its kernels (the `PhaseTimer` /
 * `GpuTiming` GPU timestamps of the struct Gpu page, here CUDA events):
 *   events  host array of MOE_PREFILL_KERNELS + 1 caller-created cudaEvent_t
 *           (as void *); events[i] is recorded on the stream before kernel i
 *           and events[MOE_PREFILL_KERNELS] after the last.  Kernels, in
 *           order: 0 prep (x^, bf16 operands, shared gate), 1 router GEMM,
 *           2 top-k, 3 per-expert counts, 4 group offsets and work lists,
 *           5 grouped row lists, 6 expert operand rows in group order,
 *           7 gate_up GEMM, 8 down GEMM, 9 bf16 output.
 * Results equal moe_prefill's. */
#define MOE_PREFILL_KERNELS 10
int moe_prefill_timed(const moe_layer *L, const float *x, int t, uint16_t *out, void *work, size_t work_bytes,
                      uint32_t *topk_idx, int *dev_status, void *const *events, moe_stream_t stream);

/* Workspace bytes moe_prefill and moe_prefill_group need for t rows (0 if the
 * arguments are invalid). */
size_t moe_prefill_workspace(const moe_layer *L, int t);

/* The routing and grouping stage of moe_prefill alone (same arguments):
 *   topk_idx   [t][top_k] uint32, topk_w [t][top_k] float32 (as moe_route)
 *   group_offs [G + 1] int32: G = n_experts (+1 when the layer has a shared
 *              expert, which is group n_experts and holds every row);
 *              group g's entries are [group_offs[g], group_offs[g+1])
 *   group_rows [t*top_k (+t)] int32: the row of each entry; inside a group
 *              rows ascend (a stable grouping)
 *   group_w    [t*top_k (+t)] float32: the entry's routing weight (shared
 *              group: the row's sigmoid gate) */
int moe_prefill_group(const moe_layer *L, const float *x, int t, uint32_t *topk_idx, float *topk_w,
                      int32_t *group_offs, int32_t *group_rows, float *group_w, void *work,
                      size_t work_bytes, int *dev_status, moe_stream_t stream);

/* Workspace bytes moe_forward needs for these layers and nb rows (0 if the
 * arguments are invalid). */
size_t moe_forward_workspace(const moe_layer *layers, int n_layers, int nb);

/* Thread-local description of the last failing host-side check or CUDA call. */
const char *moe_last_error(void);

/* ---- two-tier expert store (the `res` LRU pool and the miss counters of
 * the struct Gpu page; the module doc of the gpu.rs source page: a fixed
 * pool of slots, LRU managed, filled by reads of missing records).
 *
 * Every routed record of a layer stack lives in pinned host memory, which
 * the GPU reads directly over NVLink-C2C; the most recently used ones are
 * also cached in n_slots device-memory slots.  The store owns two device
 * tables the layers point at: expert_addr[l] (each layer's
 * moe_layer.expert_addr) and expert_tier[l] (its expert_tier).  After a
 * step, moe_tier_update takes the step's slot tables (copied back to the
 * host): the experts listed become most recently used, and the ones read
 * from host memory are copied into device slots, evicting the least
 * recently used records that step did not use.  Copies and table updates
 * run on `stream`; run the next step on the same stream.
 *
 * Ownership: host_records, slots and the two tables belong to the caller
 * and must outlive the store; host_records is registered for device access
 * here when it is not already pinned (and unregistered by destroy).
 * expert_addr == NULL makes a policy-only store: no device memory, no CUDA
 * call (the slots then have stand-in addresses after the host records). */
typedef struct moe_tier moe_tier;
typedef struct {
  int resident;               /* records in device slots */
  int last_host_reads;        /* records the last step read from host memory */
  int last_promoted;          /* of them, copied into device slots by the last update */
  long long promotions, evictions;
} moe_tier_stats;

/*   host_records host [n_layers][n_experts][stride] bytes (record of layer l, expert e)
 *   slots        device [n_slots][stride] bytes
 *   expert_addr  device [n_layers][n_experts] uint64; expert_tier device [n_layers][n_experts] uint8
 *   stride       a multiple of 256 bytes; every record starts with its 256-byte aligned layout
 * Starts with every record in host memory and the slots empty. */
int moe_tier_create(int n_layers, int n_experts, size_t stride, void *host_records, void *slots, int n_slots,
                    uint64_t *expert_addr, uint8_t *expert_tier, moe_stream_t stream, moe_tier **out);
/* slot_tab: host copy of the step's [n_layers][64] slot tables.  Returns the
 * number of records promoted (>= 0) or a negative moe_status. */
int moe_tier_update(moe_tier *t, const uint64_t *slot_tab, int n_layers, moe_stream_t stream);
/* Device slot holding (layer, expert), -1 when in host memory only, -2 for bad arguments. */
int moe_tier_slot(const moe_tier *t, int layer, int expert);
int moe_tier_get_stats(const moe_tier *t, moe_tier_stats *stats);
/* Host copy of the address table, [n_layers][n_experts] (as last uploaded). */
const uint64_t *moe_tier_addresses(const moe_tier *t);
void moe_tier_destroy(moe_tier *t);
const char *moe_tier_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_API_H */
