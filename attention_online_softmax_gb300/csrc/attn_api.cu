// C ABI of the GB300 fused-attention library: argument checks, TMA tensor-map
// encoding, work planning and kernel launches.  Declared in include/attn.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
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

// The current device must be a GB300-class part (compute capability 10.3).
attn_status check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_NO_DEVICE;
  }
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_NO_DEVICE;
  }
  if (major != 10 || minor != 3) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

// 3-D bf16 map over [heads][rows][d] with a (64 x box_rows x 1) box and the
// 128-byte swizzle that the tcgen05 operand descriptors expect.
bool encode_rows_map(CUtensorMap* map, const void* base, int d, int rows, int heads, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(rows) * d * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 4-D bf16 map over a dense bias [Bb][Hb][Nq][Nk] (Bb, Hb = 1 when broadcast);
// one box is [128 query rows][64 keys], 128-byte swizzled.  Strides in
// elements; false when the layout does not meet the TMA rules (16-byte
// aligned base and row / head / batch strides).
bool encode_bias_map(CUtensorMap* map, const void* base, int Nq, int Nk, int Hb, int Bb, long long sh,
                     long long sb) {
  auto fn = encode_fn();
  if (!fn || !aligned16(base) || Nk % 8 != 0) return false;
  const long long plane = static_cast<long long>(Nq) * Nk;
  const long long s2 = Hb > 1 ? sh : plane;
  const long long s3 = Bb > 1 ? sb : s2 * Hb;
  if (s2 % 8 != 0 || s3 % 8 != 0 || s2 <= 0 || s3 <= 0) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(Nk), static_cast<cuuint64_t>(Nq), static_cast<cuuint64_t>(Hb),
                        static_cast<cuuint64_t>(Bb)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(Nk) * 2, static_cast<cuuint64_t>(s2) * 2,
                           static_cast<cuuint64_t>(s3) * 2};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(attn::kBM), 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D bf16 map over packed queries [total_q][Hq][d]; one box is 128 tokens of
// one head x 64 columns, 128-byte swizzled (the same shared-memory image as a
// [128 rows][64 columns] box of the [B*Hq][Nq][d] layout).
bool encode_packed_q_map(CUtensorMap* map, const void* base, int d, int Hq, int total_q) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(Hq), static_cast<cuuint64_t>(total_q)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(Hq) * d * 2};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(attn::kBM)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 4-D bf16 map over the paged cache [pages][slots][Hkv][d] for the prefill
// kernel: one box is the page_size slots of one page and one KV head x 64
// columns, 128-byte swizzled, so a page lands as page_size consecutive
// 128-byte rows of a K/V tile (at a multiple of 2 KB: whole swizzle atoms).
bool encode_paged_rows_map(CUtensorMap* map, const void* base, int d, int Hkv, int page_size, int num_pages) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(Hkv),
                        static_cast<cuuint64_t>(page_size), static_cast<cuuint64_t>(num_pages)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(Hkv) * d * 2,
                           static_cast<cuuint64_t>(page_size) * Hkv * d * 2};
  cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(page_size), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 4-D bf16 map over the paged cache [pages][slots][Hkv][d]; one box is the
// [16 slots][hg heads][d] block of one page (no swizzle).
bool encode_page_map(CUtensorMap* map, const void* base, int d, int Hkv, int page_size, int num_pages, int hg) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(Hkv),
                        static_cast<cuuint64_t>(page_size), static_cast<cuuint64_t>(num_pages)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(Hkv) * d * 2,
                           static_cast<cuuint64_t>(page_size) * Hkv * d * 2};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(d), static_cast<cuuint32_t>(hg),
                       static_cast<cuuint32_t>(page_size), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
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
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
                                               cudaSuccess) {
    cudaGetLastError();
    return 148;
  }
  return n;
}

// Work counters of the persistent prefill kernel: a ring of per-launch
// [next unit, finished CTAs] pairs, zero at load time and reset to zero by the
// last CTA of the launch that used them.  Consecutive launches take
// consecutive slots, so launches in flight at the same time (up to the ring
// size, on any streams) never share a counter.
constexpr int kSchedSlots = 64;
__device__ int g_prefill_sched[kSchedSlots][2];
std::atomic<uint32_t> g_sched_seq{0};
std::mutex g_sched_mu;
int* g_sched_base[kMaxDevices] = {};

attn_status sched_slot(int** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_NO_DEVICE;
  }
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
  int* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_sched_mu);
    if (g_sched_base[dev] == nullptr) {
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_prefill_sched) != cudaSuccess || ptr == nullptr) {
        cudaGetLastError();
        return ATTN_ERR_LAUNCH;
      }
      g_sched_base[dev] = static_cast<int*>(ptr);
    }
    base = g_sched_base[dev];
  }
  *out = base + 2 * (g_sched_seq.fetch_add(1, std::memory_order_relaxed) % kSchedSlots);
  return ATTN_OK;
}

// (Batch, head) pairs per scheduling group of the plain prefill: at least
// `want` (enough heads for two waves of units), and groups of equal size --
// a short last group would start its longest units last and leave the end of
// the launch to a few SMs.  A divisor of BH up to twice `want` if there is
// one, else BH split into near-equal groups of about `want`.
int sched_group(int BH, int want) {
  if (want < 1) want = 1;
  if (want >= BH) return BH;
  for (int d = want; d <= 2 * want && d <= BH; ++d)
    if (BH % d == 0) return d;
  const int groups = BH / want;
  return (BH + groups - 1) / groups;
}

template <int D, int NQ, int STAGES, int BIAS = 0>
attn_status launch_prefill(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                           const CUtensorMap& mb, attn::PrefillParams p, int BH, cudaStream_t stream) {
  using L = attn::PrefillLayout<D, NQ, STAGES, attn::bias_slots<BIAS>(), attn::psep_path<BIAS, false>()>;
  auto kern = attn::prefill_fwd_kernel<D, NQ, STAGES, BIAS>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_LAUNCH;
  }
  p.n_units = (p.Nq + attn::kBM * NQ - 1) / (attn::kBM * NQ);
  const int sms = sm_count();
  p.group = sched_group(BH, (2 * sms + p.n_units - 1) / p.n_units);
  const long long units = static_cast<long long>(p.n_units) * BH;
  if (units > 0x7FFFFFFFLL) return ATTN_ERR_UNSUPPORTED;
  const attn_status st = sched_slot(&p.sched);
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
  using L = attn::PrefillLayout<D, NQ, STAGES, 0, attn::psep_path<0, true>()>;
  auto kern = attn::prefill_fwd_kernel<D, NQ, STAGES, 0, true>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_LAUNCH;
  }
  const attn_status st = sched_slot(&p.sched);
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
  int hg = 1;
  int chunk = attn::kChunkMax;
  int n_splits = 1;
  size_t ws_o_floats = 0;
  size_t ws_bytes = 0;
};

bool decode_plan(int num_seqs, int Hq, int Hkv, int d, int max_seqlen, DecodePlan* out) {
  if (num_seqs < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || max_seqlen < 0) return false;
  if (d != 64 && d != 128 && d != 256) return false;
  DecodePlan pl;
  for (int c : {8, 4, 2, 1}) {
    if (Hkv % c == 0 && c * d <= 1024) {
      pl.hg = c;
      break;
    }
  }
  const long long groups = static_cast<long long>(num_seqs) * (Hkv / pl.hg);
  pl.chunk = attn::kChunkMax;
  while (pl.chunk > 64 && groups * ((max_seqlen + pl.chunk - 1) / pl.chunk) < 1024) pl.chunk /= 2;
  pl.n_splits = max_seqlen > 0 ? (max_seqlen + pl.chunk - 1) / pl.chunk : 1;
  if (pl.n_splits > 1) {
    pl.ws_o_floats = static_cast<size_t>(num_seqs) * pl.n_splits * Hq * d;
    const size_t lse_floats = static_cast<size_t>(num_seqs) * pl.n_splits * Hq;
    pl.ws_bytes = ((pl.ws_o_floats + lse_floats) * 4 + 255) & ~static_cast<size_t>(255);
  }
  *out = pl;
  return true;
}

template <int D, int G>
attn_status launch_decode(const CUtensorMap& mk, const CUtensorMap& mv, attn::DecodeParams p,
                          cudaStream_t stream) {
  const int scores_bytes = p.hg * p.chunk * G * 4;
  const int fixed = scores_bytes + 2 * attn::kMaxStages * 8 + 1024;
  auto ks = attn::decode_split_kernel<D, G>;
  // Ring depth: two CTAs per SM when registers allow it (113 KB each), else
  // one CTA per SM with a deeper ring, so that enough page bytes are in flight.
  int stages = (113 * 1024 - fixed) / p.stage_bytes;
  stages = stages < 2 ? 2 : (stages > 4 ? 4 : stages);
  {
    int per_sm = 0;
    const int threads = (p.hg + 1) * 32;
    if (cudaFuncSetAttribute(ks, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024) == cudaSuccess &&
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ks, threads, stages * p.stage_bytes + fixed) ==
            cudaSuccess &&
        per_sm < 2) {
      const int deep = (200 * 1024 - fixed) / p.stage_bytes;
      stages = deep > attn::kMaxStages ? attn::kMaxStages : (deep < stages ? stages : deep);
    }
    cudaGetLastError();
  }
  p.stages = stages;
  const int smem = stages * p.stage_bytes + fixed;
  if (cudaFuncSetAttribute(ks, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_LAUNCH;
  }
  const long long gx = static_cast<long long>(p.num_seqs) * p.n_splits;
  if (gx > 0x7FFFFFFFLL) return ATTN_ERR_UNSUPPORTED;
  ks<<<dim3(static_cast<unsigned>(gx), p.Hkv / p.hg), (p.hg + 1) * 32, smem, stream>>>(mk, mv, p);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (p.n_splits > 1) {
    // Programmatic dependent launch: the combine grid is scheduled while the
    // split grid drains and waits (griddepcontrol.wait) for its partials.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.num_seqs, (p.Hq + 3) / 4);
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
    case 1: return launch_decode<D, 1>(mk, mv, p, s);
    case 2: return launch_decode<D, 2>(mk, mv, p, s);
    case 4: return launch_decode<D, 4>(mk, mv, p, s);
    case 8: return launch_decode<D, 8>(mk, mv, p, s);
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
  p.scale_log2 = scale * 1.4426950408889634f;
  p.window = mask ? mask->window_left : 0;
  p.alibi = mask ? mask->alibi_slopes : nullptr;
  p.bias = mask ? static_cast<const uint16_t*>(mask->bias) : nullptr;
  p.bias_sb = mask ? mask->bias_stride_b : 0;
  p.bias_sh = mask ? mask->bias_stride_h : 0;
  p.bias_hmul = 0;
  p.bias_bmul = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // Two query tiles per CTA (they share every K/V tile and overlap each
  // other's softmax with MMAs) unless that leaves the GPU under-filled.
  const long long pairs = static_cast<long long>((Nq + 2 * attn::kBM - 1) / (2 * attn::kBM)) * B * Hq;
  const bool two = pairs >= 2LL * sm_count();
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
        case 64: return launch_prefill<64, 1, 8, 2>(mq, mk, mv, mb, p, B * Hq, s);
        case 128: return launch_prefill<128, 1, 4, 2>(mq, mk, mv, mb, p, B * Hq, s);
        case 256: return launch_prefill<256, 1, 3, 2>(mq, mk, mv, mb, p, B * Hq, s);
        default: return ATTN_ERR_UNSUPPORTED;
      }
    }
  }
  if (p.alibi != nullptr || p.bias != nullptr) {
    // Additive-bias variants: one query tile per unit (the per-score bias
    // terms need the registers a second tile's pipeline would take).
    switch (d) {
      case 64: return launch_prefill<64, 1, 12, 1>(mq, mk, mv, mq, p, B * Hq, s);
      case 128: return launch_prefill<128, 1, 6, 1>(mq, mk, mv, mq, p, B * Hq, s);
      case 256: return launch_prefill<256, 1, 5, 1>(mq, mk, mv, mq, p, B * Hq, s);
      default: return ATTN_ERR_UNSUPPORTED;
    }
  }
  switch (d) {
    case 64:
      return two ? launch_prefill<64, 2, 10>(mq, mk, mv, mq, p, B * Hq, s)
                 : launch_prefill<64, 1, 12>(mq, mk, mv, mq, p, B * Hq, s);
    case 128:
      return two ? launch_prefill<128, 2, 4>(mq, mk, mv, mq, p, B * Hq, s)
                 : launch_prefill<128, 1, 6>(mq, mk, mv, mq, p, B * Hq, s);
    case 256: return launch_prefill<256, 1, 5>(mq, mk, mv, mq, p, B * Hq, s);
  }
  return ATTN_ERR_UNSUPPORTED;
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
      return two ? launch_prefill_paged<64, 2, 10>(mq, mk, mv, p, total_q, s)
                 : launch_prefill_paged<64, 1, 12>(mq, mk, mv, p, total_q, s);
    case 128:
      return two ? launch_prefill_paged<128, 2, 5>(mq, mk, mv, p, total_q, s)
                 : launch_prefill_paged<128, 1, 6>(mq, mk, mv, p, total_q, s);
    case 256: return launch_prefill_paged<256, 1, 5>(mq, mk, mv, p, total_q, s);
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
  if (page_size != attn::kPage) return ATTN_ERR_UNSUPPORTED;
  const int G = Hq / Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(max_seqlen) > static_cast<long long>(max_pages_per_seq) * page_size)
    return ATTN_ERR_INVALID_ARG;
  if (num_seqs == 0) return ATTN_OK;
  if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(block_table) ||
      !aligned16(seqlens) || !aligned16(o) || !aligned16(lse))
    return ATTN_ERR_MISALIGNED;
  DecodePlan pl;
  if (!decode_plan(num_seqs, Hq, Hkv, d, max_seqlen, &pl)) return ATTN_ERR_INVALID_ARG;
  if (pl.ws_bytes > 0 && (!aligned16(workspace) || workspace_bytes < pl.ws_bytes)) return ATTN_ERR_WORKSPACE;
  attn_status st = check_device();
  if (st != ATTN_OK) return st;

  CUtensorMap mk, mv;
  if (!encode_page_map(&mk, kcache, d, Hkv, page_size, num_pages, pl.hg) ||
      !encode_page_map(&mv, vcache, d, Hkv, page_size, num_pages, pl.hg))
    return ATTN_ERR_LAUNCH;

  attn::DecodeParams p;
  p.q = static_cast<const uint16_t*>(q);
  p.block_table = block_table;
  p.seqlens = seqlens;
  p.o = o;
  p.lse = lse;
  p.ws_o = static_cast<float*>(workspace);
  p.ws_lse = pl.ws_bytes > 0 ? static_cast<float*>(workspace) + pl.ws_o_floats : nullptr;
  p.num_seqs = num_seqs;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.num_pages = num_pages;
  p.max_pages = max_pages_per_seq;
  p.max_seqlen = max_seqlen;
  p.chunk = pl.chunk;
  p.n_splits = pl.n_splits;
  p.hg = pl.hg;
  p.stages = 2;
  p.stage_bytes = page_size * pl.hg * d * 2;
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
  if (chain == nullptr || out_ns == nullptr || hops <= 0 || chain_len == 0) return ATTN_ERR_INVALID_ARG;
  attn_status st = check_device();
  if (st != ATTN_OK) return st;
  attn::dram_latency_kernel<<<1, 1, 0, reinterpret_cast<cudaStream_t>(stream)>>>(chain, hops, out_ns);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return ATTN_OK;
}
