// tier.cu -- the two-tier expert store: every routed record in pinned host
// memory (Grace memory, read by the GPU over NVLink-C2C), the most recently
// used ones cached in device-memory slots.
//
// After each step the caller hands back the step's slot tables; the experts
// they list become most recently used, and those the step read from host
// memory are copied into device slots (evicting the least recently used
// records the step did not use).  The per-layer expert address and tier
// tables that the decode kernel reads are rewritten to match.  All copies
// run on the caller's stream, so the next step on that stream sees them.
//
// Sources: the `res` field (LRU expert pool) and the miss counters of the
// struct Gpu page; the module doc of the gpu.rs source page (a fixed pool
// of slots, LRU managed, filled by reads of missing records).
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <list>
#include <new>
#include <unordered_map>
#include <vector>

#include "moe_api.h"

namespace {

struct Key {
  int layer, expert;
};

}  // namespace

struct moe_tier {
  int n_layers, n_experts, n_slots;
  size_t stride;
  bool dry;                   // policy only (no device memory, no CUDA calls)
  uint8_t *host;              // caller's host records [n_layers][n_experts][stride]
  uint64_t host_dev;          // their device address (pinned, mapped)
  bool registered;            // host records registered here (unregistered at destroy)
  uint64_t slots_dev;         // device slots [n_slots][stride]
  uint64_t *addr_dev;         // device [n_layers][n_experts]
  uint8_t *tier_dev;          // device [n_layers][n_experts]
  uint64_t *addr_mirror;      // pinned host mirrors of the two tables
  uint8_t *tier_mirror;
  cudaEvent_t tables_done;    // the last table upload has read the mirrors
  std::vector<int> slot_of;   // [n_layers * n_experts] -> device slot, or -1
  std::vector<int> key_of;    // [n_slots] -> layer * n_experts + expert, or -1
  std::list<int> lru;         // resident keys, least recently used first
  std::vector<std::list<int>::iterator> pos;  // [n_layers * n_experts] position in lru
  std::vector<uint64_t> used_in;              // [n_layers * n_experts] last update that used the key
  uint64_t epoch;
  moe_tier_stats stats;
};

namespace {

thread_local char g_err[256];

int tfail(int code, const char *msg) {
  strncpy(g_err, msg, sizeof g_err - 1);
  return code;
}

// address of a record in host memory (as the device sees it) / in a slot
uint64_t host_addr(const moe_tier *t, int key) { return t->host_dev + (uint64_t)key * t->stride; }
uint64_t slot_addr(const moe_tier *t, int s) { return t->slots_dev + (uint64_t)s * t->stride; }

// the key an address listed in a slot table belongs to, or -1
int key_of_addr(const moe_tier *t, int layer, uint64_t a) {
  const uint64_t n = (uint64_t)t->n_layers * t->n_experts;
  if (a >= t->host_dev && a < t->host_dev + n * t->stride) {
    const uint64_t k = (a - t->host_dev) / t->stride;
    return (int)k / t->n_experts == layer ? (int)k : -1;
  }
  if (t->n_slots > 0 && a >= t->slots_dev && a < t->slots_dev + (uint64_t)t->n_slots * t->stride) {
    const int k = t->key_of[(a - t->slots_dev) / t->stride];
    return k >= 0 && k / t->n_experts == layer ? k : -1;
  }
  return -1;
}

void set_entry(moe_tier *t, int key, bool device, int slot) {
  t->addr_mirror[key] = device ? slot_addr(t, slot) : host_addr(t, key);
  t->tier_mirror[key] = device ? 0 : 1;
}

int upload_tables(moe_tier *t, cudaStream_t st) {
  if (t->dry) return MOE_OK;
  const size_t n = (size_t)t->n_layers * t->n_experts;
  if (cudaMemcpyAsync(t->addr_dev, t->addr_mirror, n * 8, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(t->tier_dev, t->tier_mirror, n, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaEventRecord(t->tables_done, st) != cudaSuccess)
    return tfail(MOE_ECUDA, "tier: table upload failed");
  return MOE_OK;
}

}  // namespace

extern "C" {

const char *moe_tier_last_error(void) { return g_err; }

int moe_tier_create(int n_layers, int n_experts, size_t stride, void *host_records, void *slots, int n_slots,
                    uint64_t *expert_addr, uint8_t *expert_tier, moe_stream_t stream, moe_tier **out) {
  if (!out) return tfail(MOE_EINVAL, "tier: out is NULL");
  *out = nullptr;
  if (n_layers < 1 || n_experts < 1 || n_slots < 0) return tfail(MOE_EINVAL, "tier: bad sizes");
  if (stride == 0 || stride % 256) return tfail(MOE_EALIGN, "tier: stride must be a positive multiple of 256");
  const bool dry = expert_addr == nullptr;
  if (!dry && (!host_records || !expert_tier || (n_slots > 0 && !slots)))
    return tfail(MOE_EINVAL, "tier: host_records, expert_tier and slots are needed");
  if (((uintptr_t)host_records | (uintptr_t)slots) & 255u) return tfail(MOE_EALIGN, "tier: records not 256-byte aligned");
  moe_tier *t = new (std::nothrow) moe_tier();
  if (!t) return tfail(MOE_EINVAL, "tier: out of host memory");
  const size_t n = (size_t)n_layers * n_experts;
  t->n_layers = n_layers, t->n_experts = n_experts, t->n_slots = n_slots, t->stride = stride, t->dry = dry;
  t->host = (uint8_t *)host_records;
  t->addr_dev = expert_addr, t->tier_dev = expert_tier;
  t->slots_dev = (uint64_t)(uintptr_t)slots;
  t->epoch = 0;
  memset(&t->stats, 0, sizeof t->stats);
  if (dry) {
    // policy only: addresses are the host ones, slots a stand-in range after them
    t->host_dev = (uint64_t)(uintptr_t)host_records;
    if (t->slots_dev == 0) t->slots_dev = t->host_dev + n * stride + 4096;
    t->addr_mirror = new (std::nothrow) uint64_t[n];
    t->tier_mirror = new (std::nothrow) uint8_t[n];
    if (!t->addr_mirror || !t->tier_mirror) {
      moe_tier_destroy(t);
      return tfail(MOE_EINVAL, "tier: out of host memory");
    }
  } else {
    cudaPointerAttributes at{};
    const bool pinned = cudaPointerGetAttributes(&at, host_records) == cudaSuccess && at.type == cudaMemoryTypeHost;
    if (!pinned) {
      if (cudaHostRegister(host_records, n * stride, cudaHostRegisterMapped | cudaHostRegisterReadOnly) != cudaSuccess &&
          cudaHostRegister(host_records, n * stride, cudaHostRegisterMapped) != cudaSuccess) {
        cudaGetLastError();
        delete t;
        return tfail(MOE_ECUDA, "tier: cannot register the host records for device access");
      }
      t->registered = true;
    }
    void *dp = nullptr;
    if (cudaHostGetDevicePointer(&dp, host_records, 0) != cudaSuccess ||
        cudaHostAlloc((void **)&t->addr_mirror, n * 8, cudaHostAllocDefault) != cudaSuccess ||
        cudaHostAlloc((void **)&t->tier_mirror, n, cudaHostAllocDefault) != cudaSuccess ||
        cudaEventCreateWithFlags(&t->tables_done, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      moe_tier_destroy(t);
      return tfail(MOE_ECUDA, "tier: device pointer, mirrors or event");
    }
    t->host_dev = (uint64_t)(uintptr_t)dp;
  }
  t->slot_of.assign(n, -1);
  t->key_of.assign((size_t)n_slots, -1);
  t->pos.assign(n, t->lru.end());
  t->used_in.assign(n, 0);
  for (size_t k = 0; k < n; k++) set_entry(t, (int)k, false, 0);
  const int r = upload_tables(t, (cudaStream_t)stream);
  if (r) {
    moe_tier_destroy(t);
    return r;
  }
  *out = t;
  return MOE_OK;
}

int moe_tier_update(moe_tier *t, const uint64_t *slot_tab, int n_layers, moe_stream_t stream) {
  if (!t || !slot_tab) return tfail(MOE_EINVAL, "tier: NULL argument");
  if (n_layers != t->n_layers) return tfail(MOE_EINVAL, "tier: n_layers differs from the store's");
  cudaStream_t st = (cudaStream_t)stream;
  // the mirrors may change only once the previous upload has read them
  if (!t->dry && cudaEventSynchronize(t->tables_done) != cudaSuccess) return tfail(MOE_ECUDA, "tier: event");
  const uint64_t ep = ++t->epoch;
  t->stats.last_host_reads = 0;
  t->stats.last_promoted = 0;
  std::vector<int> missed;
  for (int l = 0; l < n_layers; l++) {
    const uint64_t *row = slot_tab + (size_t)l * MOE_SLOT_STRIDE;
    for (int j = 0; j < MOE_SLOT_STRIDE - 2 && row[j] != 0; j++) {
      const int k = key_of_addr(t, l, row[j]);
      if (k < 0) return tfail(MOE_EINVAL, "tier: a slot-table address belongs to no record of that layer");
      if (t->used_in[k] == ep) continue;
      t->used_in[k] = ep;
      if (t->slot_of[k] >= 0) {
        t->lru.splice(t->lru.end(), t->lru, t->pos[k]);  // most recently used
      } else {
        missed.push_back(k);
        t->stats.last_host_reads++;
      }
    }
  }
  // promote this step's host reads, in slot-table order, while a slot is
  // free or the least recently used resident record was not used this step
  int free_slot = 0;
  for (int k : missed) {
    int s = -1;
    while (free_slot < t->n_slots && t->key_of[free_slot] >= 0) free_slot++;
    if (free_slot < t->n_slots) {
      s = free_slot;
    } else if (!t->lru.empty() && t->used_in[t->lru.front()] != ep) {
      const int victim = t->lru.front();
      t->lru.pop_front();
      t->pos[victim] = t->lru.end();
      s = t->slot_of[victim];
      t->slot_of[victim] = -1;
      set_entry(t, victim, false, 0);
      t->stats.evictions++;
    } else {
      break;  // every slot holds a record this step used
    }
    if (!t->dry &&
        cudaMemcpyAsync((void *)(uintptr_t)slot_addr(t, s), t->host + (size_t)k * t->stride, t->stride,
                        cudaMemcpyHostToDevice, st) != cudaSuccess)
      return tfail(MOE_ECUDA, "tier: record copy failed");
    t->key_of[s] = k;
    t->slot_of[k] = s;
    t->pos[k] = t->lru.insert(t->lru.end(), k);
    set_entry(t, k, true, s);
    t->stats.promotions++;
    t->stats.last_promoted++;
  }
  t->stats.resident = (int)t->lru.size();
  const int r = upload_tables(t, st);
  return r ? r : t->stats.last_promoted;
}

int moe_tier_slot(const moe_tier *t, int layer, int expert) {
  if (!t || layer < 0 || layer >= t->n_layers || expert < 0 || expert >= t->n_experts) return -2;
  return t->slot_of[(size_t)layer * t->n_experts + expert];
}

int moe_tier_get_stats(const moe_tier *t, moe_tier_stats *s) {
  if (!t || !s) return tfail(MOE_EINVAL, "tier: NULL argument");
  *s = t->stats;
  return MOE_OK;
}

const uint64_t *moe_tier_addresses(const moe_tier *t) { return t ? t->addr_mirror : nullptr; }

void moe_tier_destroy(moe_tier *t) {
  if (!t) return;
  if (t->dry) {
    delete[] t->addr_mirror;
    delete[] t->tier_mirror;
  } else {
    if (t->tables_done) {
      cudaEventSynchronize(t->tables_done);
      cudaEventDestroy(t->tables_done);
    }
    if (t->addr_mirror) cudaFreeHost(t->addr_mirror);
    if (t->tier_mirror) cudaFreeHost(t->tier_mirror);
    if (t->registered) cudaHostUnregister(t->host);
  }
  delete t;
}

}  // extern "C"
