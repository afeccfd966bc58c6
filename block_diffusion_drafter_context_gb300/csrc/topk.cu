// Top-16 candidates per mask position ("DFlash 2", Arquitectura del Sistema
// item 1: the drafter proposes a list of 16 candidates per position).
//
// Order: value descending, token id ascending on ties.  Each (value, id) is
// packed into one 64-bit key whose unsigned order is exactly that order, so
// every key is unique and the selection is deterministic.
//
// One row = the fp32 logits of one mask position over the vocabulary.  A row
// is cut into chunks, one CTA each, to fill the GPU when there are few rows.
// Every warp streams its share with 128-bit loads and keeps a sorted top-16
// in lanes 0..15; an element enters only if it beats the warp's current 16th
// key (ballot), which after the first few hundred elements almost never
// happens, so the scan runs at load speed.  Warps merge in shared memory;
// chunks merge in the CTA that finishes a row last (per-row counter).
#include "common.cuh"
#include "internal.h"

#include <mutex>

namespace dflash {
namespace {

constexpr int K = 16;
constexpr int WARPS = 8;


// Warp-wide sorted list in lanes 0..15 (descending).  Insert key k (uniform).
__device__ __forceinline__ void insert(uint64_t &list, uint64_t k, int lane) {
  const uint64_t up = __shfl_up_sync(0xffffffffu, list, 1);
  if (lane < K) list = (list > k) ? list : ((lane == 0 || up > k) ? k : up);
}

// Offer one key per lane; inserts every key that beats the current 16th.
__device__ __forceinline__ void offer(uint64_t &list, uint64_t &thr, uint64_t key, int lane) {
  unsigned m = __ballot_sync(0xffffffffu, key > thr);
  while (m) {
    const int src = __ffs(m) - 1;
    const uint64_t k = __shfl_sync(0xffffffffu, key, src);
    insert(list, k, lane);
    thr = __shfl_sync(0xffffffffu, list, K - 1);
    m &= ~(1u << src);
    m &= __ballot_sync(0xffffffffu, key > thr);
  }
}

// The 16th largest of the 32 lanes' values (a warp-wide descending bitonic
// sort; every lane gets the result).
__device__ __forceinline__ float warp_16th_largest(float v, int lane) {
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const float o = __shfl_xor_sync(0xffffffffu, v, j);
      const bool up = ((lane & k) == 0) == ((lane & j) == 0);   // this lane keeps the larger
      v = up ? fmaxf(v, o) : fminf(v, o);
    }
  }
  return __shfl_sync(0xffffffffu, v, K - 1);
}

// The end of a row's selection: this CTA's warp lists merged in shared
// memory; a row cut into chunks leaves its chunk's 16 keys in `part` and the
// CTA that completes the row last (per-row counter, self-resetting) merges
// the chunk lists.  Every warp list alone has 16 keys >= its 16th, so the
// merged 16th is at least the largest of those and smaller keys are never
// offered (the same floor between chunks).
__device__ __forceinline__ void finish_row(uint64_t list, uint64_t *sm, int &last, int row, int c, int nchunks,
                                           int32_t *ids, float *vals, uint64_t *part, int *counters) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane < K) sm[warp * K + lane] = list;
  __syncthreads();
  if (warp == 0) {
    uint64_t l2 = 0, t2 = 0, floor2 = 0;
    for (int w = 0; w < WARPS; ++w) floor2 = sm[w * K + K - 1] > floor2 ? sm[w * K + K - 1] : floor2;
    for (int i = lane; i < WARPS * K; i += 32) offer(l2, t2, sm[i] >= floor2 ? sm[i] : 0, lane);
    if (nchunks == 1) {
      if (lane < K) {
        ids[row * K + lane] = key_id(l2);
        vals[row * K + lane] = key_value(l2);
      }
    } else {
      if (lane < K) __stcg(&part[(static_cast<size_t>(row) * nchunks + c) * K + lane], l2);
      __threadfence();
      __syncwarp();
      if (lane == 0) {
        const int old = atomicAdd(&counters[row], 1);
        last = (old == nchunks - 1);
        if (last) counters[row] = 0;
        __threadfence();
      }
      __syncwarp();
      if (last) {
        const uint64_t *pr = part + static_cast<size_t>(row) * nchunks * K;
        uint64_t l3 = 0, t3 = 0, floor3 = 0;
        for (int c2 = lane; c2 < nchunks; c2 += 32) {   // the largest 16th key of the chunk lists
          const uint64_t k16 = __ldcg(&pr[c2 * K + K - 1]);
          floor3 = k16 > floor3 ? k16 : floor3;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const uint64_t t = __shfl_xor_sync(0xffffffffu, floor3, o);
          floor3 = t > floor3 ? t : floor3;
        }
        for (int i = lane; i < nchunks * K; i += 32) {
          const uint64_t k = __ldcg(&pr[i]);
          offer(l3, t3, k >= floor3 ? k : 0, lane);
        }
        if (lane < K) {
          ids[row * K + lane] = key_id(l3);
          vals[row * K + lane] = key_value(l3);
        }
      }
    }
  }
}

__global__ void __launch_bounds__(WARPS * 32) topk_kernel(const float *__restrict__ logits, int V, int chunk,
                                                          int nchunks, int32_t *ids, float *vals,
                                                          uint64_t *part, int *counters) {
  pdl_start();
  __shared__ uint64_t sm[WARPS * K];
  __shared__ int last;
  const int row = blockIdx.y, c = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float *x = logits + static_cast<size_t>(row) * V;
  const int lo = c * chunk, hi = min(V, lo + chunk);
  uint64_t list = 0, thr = 0;
  if ((V & 3) == 0) {
    // lo is a multiple of 4 (chunk is), so float4 loads stay aligned.  U
    // loads per lane are issued before any is offered: one HBM latency per
    // U x 512 bytes of a warp instead of one per 512 (the offers are cheap
    // once the list has filled, so the scan is bound by bytes in flight).
    constexpr int U = 8;
    for (int wb = lo + warp * 128; wb < hi; wb += WARPS * 128 * U) {   // warp-uniform trip count
      float4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int base = wb + u * WARPS * 128 + lane * 4;
        v[u] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        if (base < hi) v[u] = __ldcs(reinterpret_cast<const float4 *>(x + base));   // hi: a multiple of 4
      }
      // Exact pre-filter while the list fills (thr = 0, warp-uniform): 16
      // lanes hold a maximum >= tau, so the warp's 16 largest of these values
      // are all >= tau and only those are offered (the one-at-a-time inserts
      // are the expensive part of the scan).  Once the list is full its 16th
      // key filters on its own.
      float tau = -INFINITY;
      if (thr == 0) {
        float lmax = -INFINITY;
#pragma unroll
        for (int u = 0; u < U; ++u)
          lmax = fmaxf(lmax, fmaxf(fmaxf(v[u].x, v[u].y), fmaxf(v[u].z, v[u].w)));   // out of range: -inf
        tau = warp_16th_largest(lmax, lane);
      }
      // Once the list is full, a value below its 16th key's value cannot
      // enter (keys order by value first): one float compare per element and
      // one vote per four decide whether any lane builds keys at all.
      float floor_v = thr == 0 ? -INFINITY : key_value(thr);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int base = wb + u * WARPS * 128 + lane * 4;
        const bool in = base < hi;
        const float lo_v = fmaxf(tau, floor_v);
        const bool cand = in && (v[u].x >= lo_v || v[u].y >= lo_v || v[u].z >= lo_v || v[u].w >= lo_v);
        if (__any_sync(0xffffffffu, cand)) {
          offer(list, thr, in && v[u].x >= tau ? make_key(v[u].x, base) : 0, lane);
          offer(list, thr, in && v[u].y >= tau ? make_key(v[u].y, base + 1) : 0, lane);
          offer(list, thr, in && v[u].z >= tau ? make_key(v[u].z, base + 2) : 0, lane);
          offer(list, thr, in && v[u].w >= tau ? make_key(v[u].w, base + 3) : 0, lane);
          floor_v = thr == 0 ? -INFINITY : key_value(thr);
        }
      }
    }
  } else {
    for (int base = lo + warp * 32 + lane; base - lane < hi; base += WARPS * 32) {
      const bool in = base < hi;
      offer(list, thr, in ? make_key(__ldcs(x + base), base) : 0, lane);
    }
  }
  finish_row(list, sm, last, row, c, nchunks, ids, vals, part, counters);
}

// The LM head's top-16 epilogue leaves, per row, 16 sorted keys of every
// 128-row vocabulary tile; the row's top-16 is the top-16 of those keys
// (every key of the row's true top-16 is among its tile's 16 largest).
// Same chunking and merge as topk_kernel, over keys instead of logits, read
// as 16-byte pairs with U loads per lane in flight.
__global__ void __launch_bounds__(WARPS * 32) topk_merge_kernel(const uint64_t *__restrict__ cand, int n_keys,
                                                                int chunk, int nchunks, int32_t *ids, float *vals,
                                                                uint64_t *part, int *counters) {
  pdl_start();
  __shared__ uint64_t sm[WARPS * K];
  __shared__ int last;
  const int row = blockIdx.y, c = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t *x = cand + static_cast<size_t>(row) * n_keys;
  const int lo = c * chunk, hi = min(n_keys, lo + chunk);   // chunk and n_keys are even
  uint64_t list = 0, thr = 0;
  constexpr int U = 4;
  for (int wb = lo + warp * 64; wb < hi; wb += WARPS * 64 * U) {   // warp-uniform trip count
    ulonglong2 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int base = wb + u * WARPS * 64 + lane * 2;
      v[u] = base < hi ? __ldcs(reinterpret_cast<const ulonglong2 *>(x + base)) : make_ulonglong2(0ull, 0ull);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      offer(list, thr, v[u].x, lane);
      offer(list, thr, v[u].y, lane);
    }
  }
  finish_row(list, sm, last, row, c, nchunks, ids, vals, part, counters);
}

}  // namespace

int topk16(const Launch &lc, const float *logits, int rows, int V, int32_t *ids, float *vals, uint64_t *part_keys,
           int *counters, int max_chunks) {
  if (rows <= 0) return DFLASH_OK;
  if (V < K) return set_error(DFLASH_ERR_SHAPE, "top-16 needs a vocabulary of at least 16");
  // enough CTAs to cover the SMs twice, chunks of at least 4096 elements
  int nch = (2 * lc.num_sms + rows - 1) / rows;
  nch = nch > max_chunks ? max_chunks : nch;
  const int maxc = (V + 4095) / 4096;
  nch = nch > maxc ? maxc : nch;
  nch = nch < 1 ? 1 : nch;
  int chunk = (V + nch - 1) / nch;
  chunk = (chunk + 127) & ~127;
  nch = (V + chunk - 1) / chunk;
  dim3 grid(nch, rows);
  ProfScope ps(lc, "topk16", 4.0 * rows * V, 0.0);
  launch_pdl(topk_kernel, dim3(grid), dim3(WARPS * 32), 0, lc.stream, logits, V, chunk, nch, ids, vals, part_keys, counters);
  return cuda_check(cudaGetLastError(), "topk launch");
}

int topk16_merge(const Launch &lc, const uint64_t *cand, int rows, int tiles, int32_t *ids, float *vals,
                 uint64_t *part_keys, int *counters, int max_chunks) {
  if (rows <= 0) return DFLASH_OK;
  if (tiles <= 0 || (reinterpret_cast<uintptr_t>(cand) & 15))
    return set_error(DFLASH_ERR_ARG, "top-16 merge: candidates missing or misaligned");
  const int n_keys = tiles * K;
  // enough CTAs to cover the SMs twice, chunks of at least 2048 keys
  int nch = (2 * lc.num_sms + rows - 1) / rows;
  nch = nch > max_chunks ? max_chunks : nch;
  const int maxc = (n_keys + 2047) / 2048;
  nch = nch > maxc ? maxc : nch;
  nch = nch < 1 ? 1 : nch;
  int chunk = (n_keys + nch - 1) / nch;
  chunk = (chunk + 63) & ~63;
  nch = (n_keys + chunk - 1) / chunk;
  dim3 grid(nch, rows);
  ProfScope ps(lc, "topk16_merge", 8.0 * rows * n_keys, 0.0);
  launch_pdl(topk_merge_kernel, dim3(grid), dim3(WARPS * 32), 0, lc.stream, cand, n_keys, chunk, nch, ids, vals,
             part_keys, counters);
  return cuda_check(cudaGetLastError(), "top-16 merge launch");
}

// ---------------------------------------------------------------------------
// Allocation-free top-16 (dflash_topk16_noalloc).
//
// Some callers cannot allocate device memory at all: inference-engine plugin
// hooks that receive only their input and output buffers and run under a
// device-memory budget the engine planned in advance, where a cudaMalloc
// could fail or stall the device.  For them this entry point keeps the
// selection's scratch (per-chunk partial top-16 keys and per-row completion
// counters) in one fixed array inside the library instead of a caller
// workspace.  Limits: at most NOALLOC_MAX_ROWS rows and NOALLOC_MAX_CHUNKS
// chunks per row (4 MB + 4 KB held on every GPU that loads the library, until
// the process exits).  All calls share the array: calls that overlap on the
// GPU (different streams, no ordering between them) race on it.
namespace {

constexpr int NOALLOC_MAX_ROWS = 1024;
constexpr int NOALLOC_MAX_CHUNKS = 32;
constexpr size_t NOALLOC_CTR_BYTES = sizeof(int) * NOALLOC_MAX_ROWS;
constexpr size_t NOALLOC_KEY_BYTES = sizeof(uint64_t) * NOALLOC_MAX_ROWS * NOALLOC_MAX_CHUNKS * 16;

static __device__ __align__(256) unsigned char g_topk_scratch[NOALLOC_CTR_BYTES + NOALLOC_KEY_BYTES];

constexpr int NOALLOC_MAX_DEVICES = 64;
void *g_scratch_addr[NOALLOC_MAX_DEVICES] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (returned with
// the device ordinal).  The array's name is only a host-side stand-in; its
// device address is looked up once per device, with that device current, and
// cached (valid for the device's context: a cudaDeviceReset makes it stale).
int scratch_address(void **out, int *dev_out) {
  int dev = -1;
  if (int e = cuda_check(cudaGetDevice(&dev), "noalloc top-16: cudaGetDevice")) return e;
  *dev_out = dev;
  if (dev < 0 || dev >= NOALLOC_MAX_DEVICES)
    return set_error(DFLASH_ERR_UNSUPPORTED, "noalloc top-16: device ordinal %d beyond %d", dev, NOALLOC_MAX_DEVICES);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    if (int e = cuda_check(cudaGetSymbolAddress(&p, g_topk_scratch), "noalloc top-16: cudaGetSymbolAddress"))
      return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return DFLASH_OK;
}

}  // namespace
}  // namespace dflash

extern "C" DFLASH_API int dflash_topk16_noalloc(const float *logits, int rows, int vocab, int32_t *topk_ids, float *topk_logits,
                                     dflash_stream_t stream) {
  using namespace dflash;
  if (rows < 0 || vocab < 0) return set_error(DFLASH_ERR_ARG, "noalloc top-16: negative size");
  if (rows == 0) return DFLASH_OK;
  if (!logits || !topk_ids || !topk_logits) return set_error(DFLASH_ERR_ARG, "noalloc top-16: null pointer");
  if (rows > NOALLOC_MAX_ROWS)
    return set_error(DFLASH_ERR_SHAPE, "noalloc top-16: %d rows exceed the fixed scratch limit of %d rows", rows,
                     NOALLOC_MAX_ROWS);
  void *base = nullptr;
  int dev = 0;
  if (int e = scratch_address(&base, &dev)) return e;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the completion counters must start at zero; the array keeps whatever the
  // previous call left, so clear them on the stream first
  if (int e = cuda_check(cudaMemsetAsync(base, 0, sizeof(int) * rows, s), "noalloc top-16: clear counters"))
    return e;
  Launch lc;
  lc.stream = s;
  int sms = 0;
  if (int e = cuda_check(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev),
                         "noalloc top-16: SM count"))
    return e;
  if (sms > 0) lc.num_sms = sms;
  return topk16(lc, logits, rows, vocab, topk_ids, topk_logits,
                reinterpret_cast<uint64_t *>(static_cast<char *>(base) + NOALLOC_CTR_BYTES), static_cast<int *>(base),
                NOALLOC_MAX_CHUNKS);
}
