// C ABI of the GB300 fused-attention library: argument checks, TMA tensor-map
// encoding, work planning and kernel launches.  Declared in include/attn.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "attn.h"
#include "decode.cuh"
#include "prefill_fwd.cuh"
#include "ptx.cuh"

// Scratch for attn_decode_paged_static(): split partials of one call, in a
// device array owned by this library (no allocation at call time).  In host
// code the symbol is only a stand-in; its device address comes from
// cudaGetSymbolAddress, looked up once per device with that device current.
static __device__ __align__(256) unsigned char g_decode_scratch[ATTN_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::atomic<uint64_t> g_launches{0};

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// Per-device facts looked up once (the calls that query them cost host time
// on every launch otherwise): whether the device is usable here, and its SM count.
std::atomic<int> g_dev_state[kMaxDevices];  // 0 unknown, else 1 + attn_status of the check
std::atomic<int> g_dev_sms[kMaxDevices];    // 0 unknown

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  return dev;
}

// The current device must be a GB300-class part (compute capability 10.3).
attn_status check_device() {
  const int dev = current_device();
  if (dev < 0) return ATTN_ERR_NO_DEVICE;
  if (dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
  const int known = g_dev_state[dev].load(std::memory_order_relaxed);
  if (known != 0) return static_cast<attn_status>(known - 1);
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_NO_DEVICE;
  }
  const attn_status st = (major != 10 || minor != 3) ? ATTN_ERR_UNSUPPORTED : ATTN_OK;
  g_dev_state[dev].store(1 + static_cast<int>(st), std::memory_order_relaxed);
  return st;
}

// Raises a kernel's dynamic shared-memory limit to at least `bytes` on the
// current device, calling the runtime only when the limit must grow.  One
// cache per kernel (the function-local static of each Kern: the template is
// keyed by the kernel's address, not its type, which instantiations share).
template <auto Kern>
bool ensure_smem(int bytes) {
  static std::atomic<int> set_to[kMaxDevices];
  const auto kern = Kern;
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return false;
  if (set_to[dev].load(std::memory_order_relaxed) >= bytes) return true;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  int cur = set_to[dev].load(std::memory_order_relaxed);
  while (cur < bytes && !set_to[dev].compare_exchange_weak(cur, bytes, std::memory_order_relaxed)) {
  }
  return true;
}

// Tensor maps encoded for earlier calls, keyed by every argument of the
// encoding (a map depends only on them: the base address, sizes, strides, box
// and swizzle), so a repeated call on the same buffers skips the encoder.
struct MapKey {
  uint64_t v[18];
};
struct MapEntry {
  MapKey key;
  CUtensorMap map;
  bool valid;
};
constexpr int kMapCache = 64;
std::mutex g_map_mu;
MapEntry g_maps[kMapCache];
int g_map_next = 0;

bool encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base, const cuuint64_t* dims,
                  const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle swz) {
  MapKey key;
  std::memset(&key, 0, sizeof(key));
  key.v[0] = static_cast<uint64_t>(dtype) | (static_cast<uint64_t>(rank) << 8) |
             (static_cast<uint64_t>(swz) << 16);
  key.v[1] = reinterpret_cast<uintptr_t>(base);
  for (int i = 0; i < rank; ++i) {
    key.v[2 + i] = dims[i];
    key.v[7 + i] = box[i];
    if (i + 1 < rank) key.v[12 + i] = strides[i];
  }
  {
    std::lock_guard<std::mutex> lock(g_map_mu);
    for (int i = 0; i < kMapCache; ++i)
      if (g_maps[i].valid && std::memcmp(&g_maps[i].key, &key, sizeof(key)) == 0) {
        *map = g_maps[i].map;
        return true;
      }
  }
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(map, dtype, rank, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  std::lock_guard<std::mutex> lock(g_map_mu);
  MapEntry& e = g_maps[g_map_next];
  g_map_next = (g_map_next + 1) % kMapCache;
  e.key = key;
  e.map = *map;
  e.valid = true;
  return true;
}

// 3-D bf16 map over [heads][rows][d] with a (64 x box_rows x 1) box and the
// 128-byte swizzle that the tcgen05 operand descriptors expect.
bool encode_rows_map(CUtensorMap* map, const void* base, int d, int rows, int heads, int box_rows) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(rows) * d * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// 4-D bf16 map over a dense bias [Bb][Hb][Nq][Nk] (Bb, Hb = 1 when broadcast);
// one box is [128 query rows][64 keys], 128-byte swizzled.  Strides in
// elements; false when the layout does not meet the TMA rules (16-byte
// aligned base and row / head / batch strides).
bool encode_bias_map(CUtensorMap* map, const void* base, int Nq, int Nk, int Hb, int Bb, long long sh,
                     long long sb) {
  if (!aligned16(base) || Nk % 8 != 0) return false;
  const long long plane = static_cast<long long>(Nq) * Nk;
  const long long s2 = Hb > 1 ? sh : plane;
  const long long s3 = Bb > 1 ? sb : s2 * Hb;
  if (s2 % 8 != 0 || s3 % 8 != 0 || s2 <= 0 || s3 <= 0) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(Nk), static_cast<cuuint64_t>(Nq), static_cast<cuuint64_t>(Hb),
                        static_cast<cuuint64_t>(Bb)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(Nk) * 2, static_cast<cuuint64_t>(s2) * 2,
                           static_cast<cuuint64_t>(s3) * 2};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(attn::kBM), 1, 1};
  return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// 3-D bf16 map over packed queries [total_q][Hq][d]; one box is 128 tokens of
// one head x 64 columns, 128-byte swizzled (the same shared-memory image as a
// [128 rows][64 columns] box of the [B*Hq][Nq][d] layout).
bool encode_packed_q_map(CUtensorMap* map, const void* base, int d, int Hq, int total_q) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(Hq), static_cast<cuuint64_t>(total_q)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(Hq) * d * 2};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(attn::kBM)};
  return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// 4-D bf16 map over the paged cache [pages][slots][Hkv][d] for the prefill
// kernel: one box is the page_size slots of one page and one KV head x 64
// columns, 128-byte swizzled, so a page lands as page_size consecutive
// 128-byte rows of a K/V tile (at a multiple of 2 KB: whole swizzle atoms).
bool encode_paged_rows_map(CUtensorMap* map, const void* base, int d, int Hkv, int page_size, int num_pages) {
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(Hkv),
                        static_cast<cuuint64_t>(page_size), static_cast<cuuint64_t>(num_pages)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(Hkv) * d * 2,
                           static_cast<cuuint64_t>(page_size) * Hkv * d * 2};
  cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(page_size), 1};
  return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// 4-D bf16 map over the paged cache [pages][slots][Hkv][d]; one box is the
// [16 slots][hg heads][d] block of one page at a slot offset (no swizzle).
bool encode_page_map(CUtensorMap* map, const void* base, int d, int Hkv, int page_size, int num_pages, int hg) {
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(Hkv),
                        static_cast<cuuint64_t>(page_size), static_cast<cuuint64_t>(num_pages)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(Hkv) * d * 2,
                           static_cast<cuuint64_t>(page_size) * Hkv * d * 2};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(d), static_cast<cuuint32_t>(hg),
                       static_cast<cuuint32_t>(attn::kBox), 1};
  return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

// One thread waits on a barrier with two expected arrivals after only one
// arrived: the phase can never complete, so the bounded wait must give up.
__global__ void selftest_wait_kernel(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    attn::mbar_init(&bar, 2);
    attn::fence_mbar_init();
    attn::mbar_arrive(&bar);
    attn::mbar_wait_for(&bar, 0, limit_ns, 99);
  }
}

int sm_count() {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return 148;
  int n = g_dev_sms[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return 148;
  }
  g_dev_sms[dev].store(n, std::memory_order_relaxed);
  return n;
}

// Work counters of the persistent prefill kernels: a ring of 64-bit words,
// (owner tag << 32) | fetches, free (0) at load time.  Each launch gets the
// next slot and a nonzero tag of its own; its first fetch claims the word and
// its last fetch frees it (attn::sched_fetch).  Launches on different slots
// never interact; a launch whose slot is still held by an earlier one (64
// launches before it, or one replayed from a graph) waits until that launch
// has handed out its last unit, bounded (ATTN_ERR_TIMEOUT).
constexpr int kSchedSlots = 64;
__device__ unsigned long long g_prefill_sched[kSchedSlots];
std::atomic<uint32_t> g_sched_seq{0};
std::mutex g_sched_mu;
unsigned long long* g_sched_base[kMaxDevices] = {};

attn_status sched_slot(unsigned long long** out, unsigned* tag) {
  const int dev = current_device();
  if (dev < 0) return ATTN_ERR_NO_DEVICE;
  if (dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
  unsigned long long* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_sched_mu);
    if (g_sched_base[dev] == nullptr) {
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_prefill_sched) != cudaSuccess || ptr == nullptr) {
        cudaGetLastError();
        return ATTN_ERR_LAUNCH;
      }
      g_sched_base[dev] = static_cast<unsigned long long*>(ptr);
    }
    base = g_sched_base[dev];
  }
  const uint32_t seq = g_sched_seq.fetch_add(1, std::memory_order_relaxed);
  *out = base + seq % kSchedSlots;
  *tag = seq % 0xFFFFFFFFu + 1u;  // never 0 (the free word)
  return ATTN_OK;
}

// (Batch, head) pairs per scheduling group of the plain prefill: at least
// `want` (enough heads for two waves of units) unless that exceeds `cap`
// (the most heads whose K/V stays in L2, so that each K/V tile comes from
// DRAM once), and groups of equal size -- a short last group would start its
// longest units last and leave the end of the launch to a few SMs.  A
// divisor of BH from `want` up to twice `want` (and `cap`) if there is one,
// else BH split into near-equal groups of about `want`, or of at most `cap`.
int sched_group(int BH, int want, int cap) {
  if (cap < 1) cap = 1;
  if (want < 1) want = 1;
  if (want > cap) want = cap;
  if (want >= BH) return BH;
  for (int d = want; d <= 2 * want && d <= cap && d <= BH; ++d)
    if (BH % d == 0) return d;
  int groups = BH / want;
  int g = (BH + groups - 1) / groups;
  if (g > cap) {
    groups = (BH + cap - 1) / cap;
    g = (BH + groups - 1) / groups;
  }
  return g;
}

// K/V ring depth of each prefill instantiation, by head dim, query tiles per
// unit and variant (plain, additive bias read directly, staged dense bias,
// paged).  The launches below and attn_fwd_kernel_name() both read it.
constexpr int fwd_stages(int d, int nq, int bias, bool paged) {
  return paged ? (d == 64 ? (nq == 2 ? 10 : 12) : d == 128 ? (nq == 2 ? 4 : 6) : 5)
         : bias == 2 ? (d == 64 ? 8 : d == 128 ? 4 : 3)
         : bias == 1 ? (d == 64 ? 12 : d == 128 ? 6 : 5)
                     : (d == 64 ? (nq == 2 ? 10 : 12) : d == 128 ? (nq == 2 ? 4 : 6) : 5);
}

// Two query tiles per unit (they share every K/V tile and overlap each
// other's softmax with MMAs) for d <= 128 unless that leaves fewer than two
// units per SM.
bool fwd_two_tiles(long long rows_per_head, long long heads, int d) {
  if (d > 128) return false;
  return ((rows_per_head + 2 * attn::kBM - 1) / (2 * attn::kBM)) * heads >= 2LL * sm_count();
}

template <int D, int NQ, int STAGES, int BIAS = 0>
attn_status launch_prefill(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                           const CUtensorMap& mb, attn::PrefillParams p, int BH, cudaStream_t stream) {
  using L = attn::PrefillLayout<D, NQ, STAGES, attn::bias_slots<BIAS>(), attn::psep_path<BIAS, false>()>;
  auto kern = attn::prefill_fwd_kernel<D, NQ, STAGES, BIAS>;
  if (!ensure_smem<attn::prefill_fwd_kernel<D, NQ, STAGES, BIAS>>(L::kAlloc)) return ATTN_ERR_LAUNCH;
  p.n_units = (p.Nq + attn::kBM * NQ - 1) / (attn::kBM * NQ);
  const int sms = sm_count();
  // K/V bytes per query head of a group (consecutive query heads share
  // their kv head): groups hold at most ~40 MB of K/V.
  const long long kv_per_head =
      std::max(1LL, 4LL * p.Nk * D / std::max(1, p.Hq / std::max(1, p.Hkv)));
  const long long cap = std::max(1LL, std::min<long long>(BH, (40LL << 20) / kv_per_head));
  p.group = sched_group(BH, (2 * sms + p.n_units - 1) / p.n_units, static_cast<int>(cap));
  const long long units = static_cast<long long>(p.n_units) * BH;
  if (units > 0x7FFFFFFFLL) return ATTN_ERR_UNSUPPORTED;
  const attn_status st = sched_slot(&p.sched, &p.sched_tag);
  if (st != ATTN_OK) return st;
  // Persistent: one CTA per SM (or fewer when there are fewer units).
  const unsigned grid = static_cast<unsigned>(units < sms ? units : sms);
  kern<<<dim3(grid), L::kThreads, L::kAlloc, stream>>>(mq, mk, mv, mb, p);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return ATTN_OK;
}

// Paged chunked prefill: the plan kernel writes the unit prefix sums into the
// workspace, then the persistent prefill kernel (one CTA per SM) takes units
// up to the total it finds there.
template <int D, int NQ, int STAGES>
attn_status launch_prefill_paged(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                                 attn::PrefillParams p, int total_q, cudaStream_t stream) {
  using L = attn::PrefillLayout<D, NQ, STAGES, 0, attn::psep_path<0, true>(), attn::producer_warps<true>()>;
  auto kern = attn::prefill_fwd_kernel<D, NQ, STAGES, 0, true>;
  if (!ensure_smem<attn::prefill_fwd_kernel<D, NQ, STAGES, 0, true>>(L::kAlloc)) return ATTN_ERR_LAUNCH;
  const attn_status st = sched_slot(&p.sched, &p.sched_tag);
  if (st != ATTN_OK) return st;
  attn::paged_plan_kernel<<<1, 1024, 0, stream>>>(p.cu_q, p.seqlens_k, p.num_seqs, total_q, p.Hq, p.max_pages,
                                                   p.page_size, attn::kBM * NQ,
                                                   const_cast<int32_t*>(p.unit_prefix),
                                                   const_cast<int32_t*>(p.seq_order));
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  kern<<<dim3(static_cast<unsigned>(sm_count())), L::kThreads, L::kAlloc, stream>>>(mq, mk, mv, mv, p);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return ATTN_OK;
}

// ---------------------------------------------------------------- decode plan
struct DecodePlan {
  int gw = 1;   // query heads per compute warp
  int wph = 1;  // compute warps per key/value head
  int hg = 1;   // key/value heads per CTA
  int chunk = attn::kChunkMax;
  int n_splits = 1;
  size_t ws_o_floats = 0;
  size_t ws_bytes = 0;
};

bool decode_plan(int num_seqs, int Hq, int Hkv, int d, int max_seqlen, DecodePlan* out) {
  if (num_seqs < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || max_seqlen < 0) return false;
  if (d != 64 && d != 128 && d != 256) return false;
  const int G = Hq / Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) return false;
  DecodePlan pl;
  pl.gw = G < 8 ? G : 8;
  pl.wph = G / pl.gw;
  for (int c : {8, 4, 2, 1}) {
    if (Hkv % c == 0 && c * pl.wph <= 8 && c * d <= 1024) {
      pl.hg = c;
      break;
    }
  }
  const long long groups = static_cast<long long>(num_seqs) * (Hkv / pl.hg);
  pl.chunk = attn::kChunkMax;
  while (pl.chunk > 64 && groups * ((max_seqlen + pl.chunk - 1) / pl.chunk) < 1024) pl.chunk /= 2;
  pl.n_splits = max_seqlen > 0 ? (max_seqlen + pl.chunk - 1) / pl.chunk : 1;
  if (static_cast<long long>(num_seqs) * pl.n_splits > 0x7FFFFFFFLL) return false;
  if (pl.n_splits > 1) {
    pl.ws_o_floats = static_cast<size_t>(num_seqs) * pl.n_splits * Hq * d;
    const size_t lse_floats = static_cast<size_t>(num_seqs) * pl.n_splits * Hq;
    pl.ws_bytes = ((pl.ws_o_floats + lse_floats) * 4 + 255) & ~static_cast<size_t>(255);
  }
  *out = pl;
  return true;
}

// Blocks of `Kern` that fit on one SM with `smem` bytes of dynamic shared
// memory (0 when the query fails).
template <auto Kern>
int blocks_per_sm(int threads, int smem) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, Kern, threads, smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

// Ring depth of the split kernel: two CTAs per SM when the registers allow it
// and two rings of at least two stages fit (113 KB of shared memory each),
// else one CTA per SM with a deeper ring; either way enough page bytes are in
// flight to keep HBM busy.  The answer for the last shape asked on each
// device is kept (one cache per kernel).
template <auto Kern>
bool decode_stages(int threads, int fixed, int stage_bytes, int* stages) {
  constexpr int kTwo = 113 * 1024, kOne = 220 * 1024;
  struct Shape {
    int threads, fixed, stage_bytes, stages;
  };
  static std::mutex mu;
  static Shape last[kMaxDevices];
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return false;
  {
    std::lock_guard<std::mutex> lock(mu);
    const Shape& c = last[dev];
    if (c.stages > 0 && c.threads == threads && c.fixed == fixed && c.stage_bytes == stage_bytes) {
      *stages = c.stages;
      return true;
    }
  }
  if (!ensure_smem<Kern>(kOne)) return false;
  int st2 = (kTwo - fixed) / stage_bytes;
  if (st2 > attn::kMaxStages) st2 = attn::kMaxStages;
  if (st2 >= 2 && blocks_per_sm<Kern>(threads, st2 * stage_bytes + fixed) >= 2) {
    *stages = st2;
  } else {
    int st1 = (kOne - fixed) / stage_bytes;
    if (st1 > attn::kMaxStages) st1 = attn::kMaxStages;
    if (st1 < 2) return false;
    *stages = st1;
  }
  std::lock_guard<std::mutex> lock(mu);
  last[dev] = Shape{threads, fixed, stage_bytes, *stages};
  return true;
}

template <int D, int GW, int WPH>
attn_status launch_decode(const CUtensorMap& mk, const CUtensorMap& mv, attn::DecodeParams p, cudaStream_t stream) {
  constexpr auto ks = attn::decode_split_kernel<D, GW, WPH>;
  const int nw = p.hg * WPH;
  const int threads = (nw + 1) * 32;
  // scores, the ring's barriers and the slack for aligning the base
  const int fixed = nw * p.chunk * GW * 4 + 2 * attn::kMaxStages * 8 + 1024;
  int stages = 0;
  if (!decode_stages<ks>(threads, fixed, p.stage_bytes, &stages)) return ATTN_ERR_LAUNCH;
  p.stages = stages;
  const int smem = stages * p.stage_bytes + fixed;
  const long long gx = static_cast<long long>(p.num_seqs) * p.n_splits;
  if (gx > 0x7FFFFFFFLL) return ATTN_ERR_UNSUPPORTED;
  ks<<<dim3(static_cast<unsigned>(gx), p.Hkv / p.hg), threads, smem, stream>>>(mk, mv, p);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (p.n_splits > 1) {
    // Programmatic dependent launch: the combine grid is scheduled while the
    // split grid drains and waits (griddepcontrol.wait) for its partials.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.num_seqs, p.Hq);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, attn::decode_combine_kernel<D>, p) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_LAUNCH;
    }
    g_launches.fetch_add(1, std::memory_order_relaxed);
  }
  return ATTN_OK;
}

template <int D>
attn_status launch_decode_g(int G, const CUtensorMap& mk, const CUtensorMap& mv, const attn::DecodeParams& p,
                            cudaStream_t s) {
  switch (G) {
    case 1: return launch_decode<D, 1, 1>(mk, mv, p, s);
    case 2: return launch_decode<D, 2, 1>(mk, mv, p, s);
    case 4: return launch_decode<D, 4, 1>(mk, mv, p, s);
    case 8: return launch_decode<D, 8, 1>(mk, mv, p, s);
    case 16: return launch_decode<D, 8, 2>(mk, mv, p, s);
    default: return ATTN_ERR_UNSUPPORTED;
  }
}

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

attn_status static_scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_NO_DEVICE;
  }
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return ATTN_ERR_LAUNCH;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return ATTN_OK;
}

}  // namespace

namespace {
// Bytes of the paged prefill's unit prefix sums in its workspace (then the
// sequences' dispatch order).
size_t paged_prefix_bytes(int num_seqs) {
  return ((static_cast<size_t>(num_seqs) + 1) * sizeof(int32_t) + 255) & ~static_cast<size_t>(255);
}
}  // namespace

extern "C" {

int attn_abi_version(void) { return 1; }

uint64_t attn_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char* attn_status_string(attn_status s) {
  switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATTN_ERR_MISALIGNED: return "null or misaligned pointer";
    case ATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case ATTN_ERR_LAUNCH: return "kernel launch failed";
    case ATTN_ERR_TIMEOUT: return "device wait timed out";
    case ATTN_ERR_BOUNDS: return "block table entry or sequence length out of range";
    case ATTN_ERR_NO_DEVICE: return "no usable CUDA device";
  }
  return "unknown status";
}

attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                     int Nq, int Nk, int d, int causal, float scale, attn_dtype o_dtype, attn_stream_t stream) {
  return attn_fwd_masked(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, causal, scale, nullptr, o_dtype, stream);
}

attn_status attn_fwd_masked(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                            int Hkv, int Nq, int Nk, int d, int causal, float scale, const attn_mask* mask,
                            attn_dtype o_dtype, attn_stream_t stream) {
  if (mask != nullptr) {
    if (mask->window_left < 0 || mask->bias_stride_b < 0 || mask->bias_stride_h < 0) return ATTN_ERR_INVALID_ARG;
    if ((mask->alibi_slopes != nullptr && (reinterpret_cast<uintptr_t>(mask->alibi_slopes) & 3u) != 0) ||
        (mask->bias != nullptr && (reinterpret_cast<uintptr_t>(mask->bias) & 3u) != 0))
      return ATTN_ERR_MISALIGNED;
  }
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Nq < 0 || Nk < 0) return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (o_dtype != ATTN_BF16 && o_dtype != ATTN_F32) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Hq > 0x7FFFFFFFLL || static_cast<long long>(B) * Hkv > 0x7FFFFFFFLL)
    return ATTN_ERR_UNSUPPORTED;
  if (B == 0 || Nq == 0) return ATTN_OK;  // empty output
  if (!aligned16(q) || !aligned16(o) || !aligned16(lse)) return ATTN_ERR_MISALIGNED;
  if (Nk > 0 && (!aligned16(k) || !aligned16(v))) return ATTN_ERR_MISALIGNED;
  attn_status st = check_device();
  if (st != ATTN_OK) return st;

  CUtensorMap mq, mk, mv;
  // With Nk == 0 no key tile is ever loaded; the K/V maps then describe q.
  const void* kb = Nk > 0 ? k : q;
  const void* vb = Nk > 0 ? v : q;
  const int nk_map = Nk > 0 ? Nk : 1;
  const int bhkv = Nk > 0 ? B * Hkv : 1;
  if (!encode_rows_map(&mq, q, d, Nq, B * Hq, attn::kBM) ||
      !encode_rows_map(&mk, kb, d, nk_map, bhkv, 128) || !encode_rows_map(&mv, vb, d, nk_map, bhkv, 128))
    return ATTN_ERR_LAUNCH;

  attn::PrefillParams p;
  p.o = o;
  p.lse = lse;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Nq = Nq;
  p.Nk = Nk;
  p.causal = causal ? 1 : 0;
  p.o_f32 = o_dtype == ATTN_F32 ? 1 : 0;
  p.n_units = 0;
  p.group = 1;
  p.sched = nullptr;
  p.sched_tag = 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.window = mask ? mask->window_left : 0;
  p.alibi = mask ? mask->alibi_slopes : nullptr;
  p.bias = mask ? static_cast<const uint16_t*>(mask->bias) : nullptr;
  p.bias_sb = mask ? mask->bias_stride_b : 0;
  p.bias_sh = mask ? mask->bias_stride_h : 0;
  p.bias_hmul = 0;
  p.bias_bmul = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool two = fwd_two_tiles(Nq, static_cast<long long>(B) * Hq, d);
  if (p.bias != nullptr && Nk > 0) {
    // A dense bias whose layout TMA can tile is staged into shared memory by
    // the producer (coalesced, asynchronous); any other layout is read by the
    // softmax threads directly.
    const int Hb = p.bias_sh != 0 ? Hq : 1;
    const int Bb = p.bias_sb != 0 ? B : 1;
    CUtensorMap mb;
    if (encode_bias_map(&mb, p.bias, Nq, Nk, Hb, Bb, p.bias_sh, p.bias_sb)) {
      p.bias_hmul = Hb > 1 ? 1 : 0;
      p.bias_bmul = Bb > 1 ? 1 : 0;
      switch (d) {
        case 64: return launch_prefill<64, 1, fwd_stages(64, 1, 2, false), 2>(mq, mk, mv, mb, p, B * Hq, s);
        case 128: return launch_prefill<128, 1, fwd_stages(128, 1, 2, false), 2>(mq, mk, mv, mb, p, B * Hq, s);
        case 256: return launch_prefill<256, 1, fwd_stages(256, 1, 2, false), 2>(mq, mk, mv, mb, p, B * Hq, s);
        default: return ATTN_ERR_UNSUPPORTED;
      }
    }
  }
  if (p.alibi != nullptr || p.bias != nullptr) {
    // Additive-bias variants: one query tile per unit (the per-score bias
    // terms need the registers a second tile's pipeline would take).
    switch (d) {
      case 64: return launch_prefill<64, 1, fwd_stages(64, 1, 1, false), 1>(mq, mk, mv, mq, p, B * Hq, s);
      case 128: return launch_prefill<128, 1, fwd_stages(128, 1, 1, false), 1>(mq, mk, mv, mq, p, B * Hq, s);
      case 256: return launch_prefill<256, 1, fwd_stages(256, 1, 1, false), 1>(mq, mk, mv, mq, p, B * Hq, s);
      default: return ATTN_ERR_UNSUPPORTED;
    }
  }
  switch (d) {
    case 64:
      return two ? launch_prefill<64, 2, fwd_stages(64, 2, 0, false)>(mq, mk, mv, mq, p, B * Hq, s)
                 : launch_prefill<64, 1, fwd_stages(64, 1, 0, false)>(mq, mk, mv, mq, p, B * Hq, s);
    case 128:
      return two ? launch_prefill<128, 2, fwd_stages(128, 2, 0, false)>(mq, mk, mv, mq, p, B * Hq, s)
                 : launch_prefill<128, 1, fwd_stages(128, 1, 0, false)>(mq, mk, mv, mq, p, B * Hq, s);
    case 256: return launch_prefill<256, 1, fwd_stages(256, 1, 0, false)>(mq, mk, mv, mq, p, B * Hq, s);
  }
  return ATTN_ERR_UNSUPPORTED;
}

const char* attn_fwd_kernel_name(int B, int Hq, int Nq, int d) {
  static thread_local char buf[96];
  if (B <= 0 || Hq <= 0 || Nq <= 0 || (d != 64 && d != 128 && d != 256)) return "";
  const int nq = fwd_two_tiles(Nq, static_cast<long long>(B) * Hq, d) ? 2 : 1;
  std::snprintf(buf, sizeof(buf), "prefill_fwd_kernel<%d,%d,%d,0,0>", d, nq, fwd_stages(d, nq, 0, false));
  return buf;
}

size_t attn_prefill_paged_workspace_size(int num_seqs) {
  if (num_seqs < 0) return 0;
  // Unit prefix sums, then the sequences' dispatch order.
  return paged_prefix_bytes(num_seqs) +
         ((static_cast<size_t>(num_seqs) * sizeof(int32_t) + 255) & ~static_cast<size_t>(255));
}

attn_status attn_prefill_paged(const void* q, const void* kcache, const void* vcache, const int32_t* block_table,
                               const int32_t* cu_seqlens_q, const int32_t* seqlens_k, void* o, float* lse,
                               int num_seqs, int total_q, int Hq, int Hkv, int d, int page_size, int num_pages,
                               int max_pages_per_seq, int causal, int window_left, float scale, void* workspace,
                               size_t workspace_bytes, attn_dtype o_dtype, attn_stream_t stream) {
  if (num_seqs < 0 || total_q < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (num_pages <= 0 || max_pages_per_seq <= 0 || window_left < 0) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (o_dtype != ATTN_BF16 && o_dtype != ATTN_F32) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return ATTN_ERR_UNSUPPORTED;
  if (page_size != 16 && page_size != 32 && page_size != 64 && page_size != 128) return ATTN_ERR_UNSUPPORTED;
  if ((static_cast<long long>(total_q) + attn::kBM - 1) / attn::kBM * Hq > 0x7FFFFFFFLL) return ATTN_ERR_UNSUPPORTED;
  if (num_seqs == 0 || total_q == 0) return ATTN_OK;
  if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(o) || !aligned16(lse))
    return ATTN_ERR_MISALIGNED;
  if (block_table == nullptr || cu_seqlens_q == nullptr || seqlens_k == nullptr) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(workspace) || workspace_bytes < attn_prefill_paged_workspace_size(num_seqs))
    return ATTN_ERR_WORKSPACE;
  attn_status st = check_device();
  if (st != ATTN_OK) return st;

  CUtensorMap mq, mk, mv;
  if (!encode_packed_q_map(&mq, q, d, Hq, total_q) ||
      !encode_paged_rows_map(&mk, kcache, d, Hkv, page_size, num_pages) ||
      !encode_paged_rows_map(&mv, vcache, d, Hkv, page_size, num_pages))
    return ATTN_ERR_LAUNCH;

  attn::PrefillParams p;
  std::memset(&p, 0, sizeof(p));
  p.o = o;
  p.lse = lse;
  p.B = 1;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.causal = causal ? 1 : 0;
  p.o_f32 = o_dtype == ATTN_F32 ? 1 : 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.window = window_left;
  p.cu_q = cu_seqlens_q;
  p.seqlens_k = seqlens_k;
  p.block_table = block_table;
  p.unit_prefix = static_cast<const int32_t*>(workspace);
  p.seq_order = reinterpret_cast<const int32_t*>(static_cast<uint8_t*>(workspace) + paged_prefix_bytes(num_seqs));
  p.num_seqs = num_seqs;
  p.max_pages = max_pages_per_seq;
  p.page_size = page_size;
  p.num_pages = num_pages;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // Two query tiles per unit (halving the page boxes per query row) when the
  // packed rows still give at least two such units per SM (an upper bound on
  // the unit count: sequences are ragged, only the total is known here).
  const bool two = (static_cast<long long>(total_q) / (2 * attn::kBM)) * Hq >= 2LL * sm_count();
  switch (d) {
    case 64:
      return two ? launch_prefill_paged<64, 2, fwd_stages(64, 2, 0, true)>(mq, mk, mv, p, total_q, s)
                 : launch_prefill_paged<64, 1, fwd_stages(64, 1, 0, true)>(mq, mk, mv, p, total_q, s);
    case 128:
      return two ? launch_prefill_paged<128, 2, fwd_stages(128, 2, 0, true)>(mq, mk, mv, p, total_q, s)
                 : launch_prefill_paged<128, 1, fwd_stages(128, 1, 0, true)>(mq, mk, mv, p, total_q, s);
    case 256: return launch_prefill_paged<256, 1, fwd_stages(256, 1, 0, true)>(mq, mk, mv, p, total_q, s);
  }
  return ATTN_ERR_UNSUPPORTED;
}

size_t attn_decode_workspace_size(int num_seqs, int Hq, int Hkv, int d, int max_seqlen) {
  DecodePlan pl;
  if (!decode_plan(num_seqs, Hq, Hkv, d, max_seqlen, &pl)) return 0;
  return pl.ws_bytes;
}

attn_status attn_decode_paged(const void* q, const void* kcache, const void* vcache, const int32_t* block_table,
                              const int32_t* seqlens, void* o, float* lse, int num_seqs, int Hq, int Hkv, int d,
                              int page_size, int num_pages, int max_pages_per_seq, int max_seqlen, float scale,
                              void* workspace, size_t workspace_bytes, attn_dtype o_dtype, attn_stream_t stream) {
  if (num_seqs < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (num_pages <= 0 || max_pages_per_seq <= 0 || max_seqlen < 0) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (o_dtype != ATTN_BF16 && o_dtype != ATTN_F32) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return ATTN_ERR_UNSUPPORTED;
  if (page_size != 16 && page_size != 32 && page_size != 64 && page_size != 128) return ATTN_ERR_UNSUPPORTED;
  const int G = Hq / Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(max_seqlen) > static_cast<long long>(max_pages_per_seq) * page_size)
    return ATTN_ERR_INVALID_ARG;
  if (num_seqs == 0) return ATTN_OK;
  if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(block_table) ||
      !aligned16(seqlens) || !aligned16(o) || !aligned16(lse))
    return ATTN_ERR_MISALIGNED;
  DecodePlan pl;
  if (!decode_plan(num_seqs, Hq, Hkv, d, max_seqlen, &pl)) return ATTN_ERR_UNSUPPORTED;
  if (pl.ws_bytes > 0 && (!aligned16(workspace) || workspace_bytes < pl.ws_bytes)) return ATTN_ERR_WORKSPACE;
  attn_status st = check_device();
  if (st != ATTN_OK) return st;

  CUtensorMap mk, mv;
  if (!encode_page_map(&mk, kcache, d, Hkv, page_size, num_pages, pl.hg) ||
      !encode_page_map(&mv, vcache, d, Hkv, page_size, num_pages, pl.hg))
    return ATTN_ERR_LAUNCH;

  attn::DecodeParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = static_cast<const uint16_t*>(q);
  p.block_table = block_table;
  p.seqlens = seqlens;
  p.o = o;
  p.lse = lse;
  if (pl.ws_bytes > 0) {
    p.ws_o = static_cast<float*>(workspace);
    p.ws_lse = static_cast<float*>(workspace) + pl.ws_o_floats;
  }
  p.num_seqs = num_seqs;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.num_pages = num_pages;
  p.max_pages = max_pages_per_seq;
  p.max_seqlen = max_seqlen;
  p.page_size = page_size;
  p.chunk = pl.chunk;
  p.n_splits = pl.n_splits;
  p.hg = pl.hg;
  p.stage_bytes = attn::kBox * pl.hg * d * 2;
  p.o_f32 = o_dtype == ATTN_F32 ? 1 : 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  switch (d) {
    case 64: return launch_decode_g<64>(G, mk, mv, p, s);
    case 128: return launch_decode_g<128>(G, mk, mv, p, s);
    case 256: return launch_decode_g<256>(G, mk, mv, p, s);
  }
  return ATTN_ERR_UNSUPPORTED;
}

const char* attn_decode_kernel_name(int num_seqs, int Hq, int Hkv, int d, int max_seqlen) {
  static thread_local char buf[96];
  DecodePlan pl;
  if (num_seqs <= 0 || !decode_plan(num_seqs, Hq, Hkv, d, max_seqlen, &pl)) return "";
  std::snprintf(buf, sizeof(buf), "decode_split_kernel<%d,%d,%d>%s", d, pl.gw, pl.wph,
                pl.n_splits > 1 ? " + decode_combine_kernel" : "");
  return buf;
}

attn_status attn_decode_paged_static(const void* q, const void* kcache, const void* vcache,
                                     const int32_t* block_table, const int32_t* seqlens, void* o, float* lse,
                                     int num_seqs, int Hq, int Hkv, int d, int page_size, int num_pages,
                                     int max_pages_per_seq, int max_seqlen, float scale, attn_dtype o_dtype,
                                     attn_stream_t stream) {
  // Too large for the built-in scratch: refuse before touching the device.
  const size_t need = attn_decode_workspace_size(num_seqs, Hq, Hkv, d, max_seqlen);
  if (need > static_cast<size_t>(ATTN_STATIC_SCRATCH_BYTES)) return ATTN_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    const attn_status st = static_scratch_address(&scratch);
    if (st != ATTN_OK) return st;
  }
  return attn_decode_paged(q, kcache, vcache, block_table, seqlens, o, lse, num_seqs, Hq, Hkv, d, page_size,
                           num_pages, max_pages_per_seq, max_seqlen, scale, scratch,
                           static_cast<size_t>(ATTN_STATIC_SCRATCH_BYTES), o_dtype, stream);
}

attn_status attn_selftest_wait_timeout(uint32_t limit_us, attn_stream_t stream) {
  if (limit_us < 1 || limit_us > 1000000) return ATTN_ERR_INVALID_ARG;
  attn_status st = check_device();
  if (st != ATTN_OK) return st;
  selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<uint64_t>(limit_us) * 1000ull);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return ATTN_OK;
}

attn_status attn_get_device_status(attn_stream_t stream) {
  attn_status st = check_device();
  if (st != ATTN_OK) return st;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_LAUNCH;
  }
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, attn::g_status, sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_LAUNCH;
  }
  const int zero = 0;
  if (cudaMemcpyToSymbol(attn::g_status, &zero, sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_LAUNCH;
  }
  return static_cast<attn_status>(v);
}

}  // extern "C"

#include "bwd_api.cuh"
#include "probe.cuh"

extern "C" attn_status attn_probe_dram_latency(const uint32_t* chain, size_t chain_len, int hops,
                                               unsigned long long* out_ns, attn_stream_t stream) {
  if (chain == nullptr || out_ns == nullptr || hops <= 0 || chain_len == 0 || chain_len > 0xFFFFFFFFull)
    return ATTN_ERR_INVALID_ARG;
  attn_status st = check_device();
  if (st != ATTN_OK) return st;
  attn::dram_latency_kernel<<<1, 1, 0, reinterpret_cast<cudaStream_t>(stream)>>>(chain, chain_len, hops, out_ns);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return ATTN_OK;
}
