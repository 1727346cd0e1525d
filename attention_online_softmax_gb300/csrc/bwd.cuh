// Attention backward: dQ, dK, dV by recomputing the weights from the saved
// row logsumexp ("Tang: a compiler that derives GPU kernels and bounds how
// fast they can run", abstract: a flash-style backward that writes no
// intermediates; the derivative of the forward of "Compilers and Kernels",
// section "FlashAttention changes the algorithm around IO").
//
// This file's kernel serves head dim 64 (bwd_wide.cuh serves 128 and 256);
// the prep and conversion kernels and the bias helpers serve all three.
// Per (batch, kv head, 128-key tile) one CTA keeps K, V, and the dK, dV
// accumulators resident and walks every (query head of the group, 128-row
// query tile) whose rows see its keys:
//   S^T  = K Q^T              (tensor memory, rows = keys)
//   P^T  = exp(scale S^T - LSE)      with the mask (0 where disallowed)
//   dP^T = V dO^T
//   dS^T = P^T * (dP^T - D),  D = rowsum(dO * O) (prep kernel)
//   dV  += P^T dO,  dK += dS^T Q     (A operands from tensor memory)
//   dQ_t = dS K                      (dS staged in shared memory), added to an
//                                     f32 dQ accumulator by TMA reduce-adds
// The 1/sqrt(d)-style scale is applied to dK at the end and to dQ as it is
// accumulated.  Roles: warp 0 TMA producer, warp 1 MMA issuer (one thread),
// warps 2..9 two per TMEM lane quarter: each thread takes one key row and half
// of the item's 128 query columns (weights, dS), then one query row and half
// of the head dim (the dQ tile's accumulation), with bounded waits everywhere.
// Each half writes its P^T and dS^T (bf16) over its own half of the dP^T
// columns, so the two threads of a key row never touch each other's columns.
#pragma once

#include "ptx.cuh"

namespace attn {

struct BwdParams {
  void* dk;            // [B*Hkv][Nk][d] bf16 or f32
  void* dv;
  float* dq_acc;       // [B*Hq][Nq][d] f32, zero on entry
  const float* lse;    // [B*Hq][Nq] forward row logsumexp (natural log)
  const float* dsum;   // [B*Hq][Nq] rowsum(dO * O) (prep kernel)
  int B, Hq, Hkv, Nq, Nk;
  int causal;
  int g_f32;           // gradients written as f32 (else bf16)
  float scale;         // > 0
  float scale_log2;    // scale * log2(e)
  int head_group;                 // (batch, kv head) pairs whose key tiles are handed out together
  // Additive bias C of the forward: the window in every instantiation, the
  // ALiBi and dense terms in the BIAS ones only.
  int window_left;                // > 0: query i keeps keys j > i + (Nk - Nq) - window_left
  const float* alibi;             // [Hq] slopes or null: C += alibi[h] (j - i - (Nk - Nq))
  const uint16_t* bias;           // bf16 or null: C += bias[b sb + h sh + i Nk + j]
  long long bias_sb, bias_sh;
};

// The bias of one query head for one key row of the backward's weight phase:
// per query column c of the item, log2(e) * C at (query q0 + c, key kj).
struct BwdBiasRow {
  float alibi_l2;        // alibi slope * log2(e) (0 without ALiBi)
  float alibi_base;      // alibi slope * log2(e) * (kj - (Nk - Nq) - q0)
  const uint16_t* brow;  // bias + b sb + h sh + q0 Nk + kj, or null
  long long bstride;     // Nk
};

__device__ __forceinline__ void prefetch_l2(const void* ptr) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
}

__device__ __forceinline__ BwdBiasRow bwd_bias_row(const BwdParams& p, int bh, int q0, int kj) {
  BwdBiasRow r;
  const int b = bh / p.Hq, h = bh - b * p.Hq;
  const float sl = p.alibi ? __ldg(p.alibi + h) * 1.4426950408889634f : 0.f;
  r.alibi_l2 = sl;
  r.alibi_base = sl * static_cast<float>(kj - (p.Nk - p.Nq) - q0);
  r.brow = p.bias ? p.bias + b * p.bias_sb + h * p.bias_sh + static_cast<long long>(q0) * p.Nk + kj : nullptr;
  r.bstride = p.Nk;
  return r;
}

// log2(e) * C at query column c of a key row (the dense bias is read only
// where the element is allowed).
__device__ __forceinline__ float bwd_bias_at(const BwdBiasRow& r, int c, bool key_ok, int c_lo, int c_hi) {
  float v = r.alibi_base - r.alibi_l2 * static_cast<float>(c);
  if (r.brow != nullptr && key_ok && c >= c_lo && c < c_hi)
    v += bf16lo(static_cast<uint32_t>(__ldg(r.brow + c * r.bstride))) * 1.4426950408889634f;
  return v;
}

// Key tile and (batch, kv head) pair of block `blk` (key-tile blocks, the
// head-dim halves of d = 256 already folded): blocks come in groups of
// head_group pairs, within a group key tile 0 first, so the pairs in flight
// at once share few heads and their Q, dO and dQ accumulator stay in L2.
__device__ __forceinline__ void bwd_block_tile(const BwdParams& p, int blk, int& kt, int& bkv) {
  const int nkt = (p.Nk + 127) / 128;
  const int BHkv = p.B * p.Hkv;
  const int gspan = p.head_group * nkt;
  const int grp = blk / gspan;
  const int in_grp = blk - grp * gspan;
  const int gcount = min(p.head_group, BHkv - grp * p.head_group);  // pairs in this (possibly smaller last) group
  kt = in_grp / gcount;
  bkv = grp * p.head_group + (in_grp - kt * gcount);
}

// Query tiles [qt_lo, qt_hi) of rows bq whose rows see some key of the key
// tile [k0, k0 + 128): causal keeps rows i >= k0 - (Nk - Nq), a left window
// rows i <= min(k0 + 127, Nk - 1) - (Nk - Nq) + window - 1.
__device__ __forceinline__ void bwd_query_tiles(const BwdParams& p, int k0, int bq, int& qt_lo, int& qt_hi) {
  const int diag = p.Nk - p.Nq;
  const int ntq = (p.Nq + bq - 1) / bq;
  qt_lo = 0;
  qt_hi = ntq;
  if (p.causal) qt_lo = max(0, (k0 - diag) / bq);
  if (p.causal && k0 - diag >= p.Nq) qt_lo = ntq;
  if (p.window_left > 0) {
    const int i_max = min(k0 + 127, p.Nk - 1) - diag + p.window_left - 1;
    qt_hi = i_max < 0 ? 0 : min(ntq, i_max / bq + 1);
  }
  if (qt_hi < qt_lo) qt_hi = qt_lo;
}

template <int D, int STAGES>
struct BwdLayout {
  static constexpr int kThreads = 320;
  static constexpr int kTile = 128 * D * 2;           // one [128][D] bf16 tile, 64-column swizzled boxes
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kTile;
  static constexpr int kQOff = kVOff + kTile;         // STAGES x (Q tile, dO tile)
  static constexpr int kStage = 2 * kTile;
  static constexpr int kDSOff = kQOff + STAGES * kStage;   // dS^T [128 keys][128 queries] bf16
  static constexpr int kDSBytes = 128 * 128 * 2;
  // 2 x (-LSE log2 e [128], D[128]) f32, one per item parity
  static constexpr int kRowOff = kDSOff + kDSBytes;
  static constexpr int kRowBytes = 2 * 128 * 4;
  static constexpr int kBarOff = kRowOff + 2 * kRowBytes;
  // kv_full, q_full[S], q_empty[S], s_full, dp_full, ds_full, dq_full, dq_free, dkv_done, rows_ready[2],
  // red_full[2], red_free[2]
  static constexpr int kNumBars = 1 + 2 * STAGES + 6 + 2 + 4;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kMiscOff + 16;
  static constexpr int kAlloc = kBytes + 128;         // the base is checked for 1024-byte alignment
  // Tensor memory columns: dK, dV accumulators, the S^T slot, the dP^T slot
  // (later, for query half h of the item, dS^T in columns [64h, 64h + 32)
  // and P^T in [64h + 32, 64h + 64)), and the dQ tile (its own columns when
  // they fit, else the S^T slot, free once S^T has been read).
  static constexpr int kColDK = 0;
  static constexpr int kColDV = D;
  static constexpr int kColS = 2 * D;
  static constexpr int kColDP = 2 * D + 128;
  static constexpr bool kSharedDQ = 3 * D + 256 > 512;
  static constexpr int kColDQ = kSharedDQ ? kColS : 2 * D + 256;
  static_assert(kBytes + 128 <= 232448, "shared memory budget");
  static_assert(D == 64 || D == 128, "backward head dims");
};

// D[r] = sum_c O[r][c] dO[r][c] (f32), d / 8 lanes per row (each lane 8
// columns, 16-byte loads), and the dQ accumulator (zero4 float4 words)
// zeroed.
__global__ void bwd_prep_kernel(const uint16_t* o, const uint16_t* dout, float* Dsum, float* dq_acc, long long rows,
                                int d, long long zero4) {
  const int lpr = d / 8;  // lanes per row: 8, 16 or 32
  const int lane = threadIdx.x & 31;
  const int sub = lane % lpr;
  const long long rows_per_warp = 32 / lpr;
  const long long nwarps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  const long long w0 = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  for (long long r0 = w0 * rows_per_warp; r0 < rows; r0 += nwarps * rows_per_warp) {
    const long long r = r0 + lane / lpr;
    float acc = 0.f;
    if (r < rows) {
      const uint4 a = *reinterpret_cast<const uint4*>(o + r * d + sub * 8);
      const uint4 b = *reinterpret_cast<const uint4*>(dout + r * d + sub * 8);
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc = fmaf(bf16lo(aw[e]), bf16lo(bw[e]), acc);
        acc = fmaf(bf16hi(aw[e]), bf16hi(bw[e]), acc);
      }
    }
    for (int off = lpr / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
    if (sub == 0 && r < rows) Dsum[r] = acc;
  }
  // From the end, so that the rows the backward's first blocks add to are the
  // ones still in L2 when it starts.
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < zero4;
       i += static_cast<long long>(gridDim.x) * blockDim.x)
    reinterpret_cast<float4*>(dq_acc)[zero4 - 1 - i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// dq = dq_acc as bf16 (RNE) or f32.  Each thread has four 16-byte loads in
// flight per round, and the rounds walk the accumulator from its end: the
// rows the backward added to last are the ones still in L2.
__global__ void bwd_post_kernel(const float* dq_acc, void* dq, long long n4, int g_f32) {
  constexpr int kU = 4;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (long long r0 = 0; r0 < n4; r0 += kU * stride) {
    float4 v[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const long long i = n4 - 1 - (r0 + u * stride + t);
      if (i >= 0) v[u] = reinterpret_cast<const float4*>(dq_acc)[i];
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const long long i = n4 - 1 - (r0 + u * stride + t);
      if (i < 0) continue;
      if (g_f32) {
        reinterpret_cast<float4*>(dq)[i] = v[u];
      } else {
        reinterpret_cast<uint2*>(dq)[i] = make_uint2(pack_bf16(v[u].x, v[u].y), pack_bf16(v[u].z, v[u].w));
      }
    }
  }
}

// out[box at (x, y, z)] += smem box, f32, by the TMA unit (rows past the
// tensor's extent are not written).
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, const void* src, int x, int y, int z) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
// global box at (x, y, z) = smem box, by the TMA unit (rows past the tensor's
// extent are not written).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N committed bulk groups of this thread still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

template <int D, int STAGES, bool BIAS>
__global__ void __launch_bounds__(320, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                    const __grid_constant__ CUtensorMap tmDQ, const BwdParams p) {
  using L = BwdLayout<D, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  if (pad + L::kBytes > static_cast<uint32_t>(L::kAlloc)) {
    // The dynamic shared memory does not start close enough to a 1024-byte
    // boundary for this layout: report instead of overrunning it.
    if (threadIdx.x == 0) report_error(5 /* ATTN_ERR_LAUNCH */, 30, static_cast<int>(pad));
    return;
  }
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw + pad;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* kv_full = bars;
  uint64_t* q_full = bars + 1;
  uint64_t* q_empty = q_full + STAGES;
  uint64_t* s_full = q_empty + STAGES;
  uint64_t* dp_full = s_full + 1;
  uint64_t* ds_full = dp_full + 1;
  uint64_t* dq_full = ds_full + 1;
  uint64_t* dq_free = dq_full + 1;
  uint64_t* dkv_done = dq_free + 1;
  uint64_t* rows_ready = dkv_done + 1;  // [2]: the item's LSE / D values are in shared memory
  // dQ tiles leave through two 16 KB staging buffers in the dS region, one
  // per half of the weight warps:
  uint64_t* red_full = rows_ready + 2;  // [2] a [128 rows][32 columns] f32 chunk is staged
  uint64_t* red_free = red_full + 2;    // [2] the TMA reduce has finished reading it
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int kt, bkv;
  bwd_block_tile(p, static_cast<int>(blockIdx.x), kt, bkv);
  const int b = bkv / p.Hkv;
  const int kvh = bkv - b * p.Hkv;
  const int k0 = kt * 128;
  const int G = p.Hq / p.Hkv;
  const int diag = p.Nk - p.Nq;
  int qt_lo, qt_hi;
  bwd_query_tiles(p, k0, 128, qt_lo, qt_hi);
  const int per_head = qt_hi - qt_lo;
  const int n_items = G * per_head;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(ds_full, 8);
    mbar_init(dq_full, 1);
    mbar_init(dq_free, 8);
    mbar_init(dkv_done, 1);
    mbar_init(&rows_ready[0], 128);
    mbar_init(&rows_ready[1], 128);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&red_full[i], 128);
      mbar_init(&red_free[i], 1);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Item n: query head bh_q = b*Hq + kvh*G + n / per_head, query tile qt_lo + n % per_head.
  auto item_bh = [&](int n) { return b * p.Hq + kvh * G + n / per_head; };
  auto item_q0 = [&](int n) { return (qt_lo + n % per_head) * 128; };

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0 && n_items > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
      mbar_expect_tx(kv_full, 2 * L::kTile);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        tma_load_3d(smem + L::kKOff + c * (128 * 128), &tmK, kv_full, c * 64, k0, bkv);
        tma_load_3d(smem + L::kVOff + c * (128 * 128), &tmV, kv_full, c * 64, k0, bkv);
      }
      int n = 0;
      for (; n < n_items; ++n) {
        const int st = n % STAGES;
        if (!mbar_wait(&q_empty[st], ((n / STAGES) & 1) ^ 1, 40)) break;
        mbar_expect_tx(&q_full[st], L::kStage);
        const int bh = item_bh(n), q0 = item_q0(n);
        uint8_t* stage = smem + L::kQOff + st * L::kStage;
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          tma_load_3d(stage + c * (128 * 128), &tmQ, &q_full[st], c * 64, q0, bh);
          tma_load_3d(stage + L::kTile + c * (128 * 128), &tmDO, &q_full[st], c * 64, q0, bh);
        }
      }
      // Drain: never leave the CTA with a copy still writing shared memory.
      mbar_wait(kv_full, 0, 41);
      for (int it = max(0, n - STAGES); it < n; ++it) mbar_wait(&q_full[it % STAGES], (it / STAGES) & 1, 42);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0 && n_items > 0) {
      constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, 0, 0);  // S^T, dP^T: K-major A and B
      constexpr uint32_t kIdG = idesc_bf16_f32(128, D, 0, 1);    // dV, dK: A from TMEM, B MN-major
      constexpr uint32_t kIdQ = idesc_bf16_f32(128, D, 1, 1);    // dQ: A (dS) and B (K) MN-major
      const uint64_t dK_a = sdesc_sw128(sbase + L::kKOff, 16, 1024);
      const uint64_t dV_a = sdesc_sw128(sbase + L::kVOff, 16, 1024);
      const uint64_t dK_b = sdesc_sw128(sbase + L::kKOff, 128 * 128, 1024);
      const uint64_t dS_a = sdesc_sw128(sbase + L::kDSOff, 128 * 128, 1024);
      bool ok = mbar_wait(kv_full, 0, 43);
      if (ok) tc_fence_after();
      for (int n = 0; ok && n < n_items; ++n) {
        const int st = n % STAGES;
        ok = mbar_wait(&q_full[st], (n / STAGES) & 1, 44);
        if (!ok) break;
        tc_fence_after();
        const uint32_t qs = sbase + L::kQOff + st * L::kStage;
        const uint64_t dQ_b = sdesc_sw128(qs, 16, 1024);
        const uint64_t dO_b = sdesc_sw128(qs + L::kTile, 16, 1024);
        const uint64_t dQ_mn = sdesc_sw128(qs, 128 * 128, 1024);
        const uint64_t dO_mn = sdesc_sw128(qs + L::kTile, 128 * 128, 1024);
        // dP^T = V dO^T (K = d) first: its slot is free once the previous
        // item's dV and dK products (issued earlier) have read it.
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t o = static_cast<uint64_t>(((kk >> 2) * (128 * 128) + (kk & 3) * 32) >> 4);
          umma_bf16_ss(tmem + L::kColDP, dV_a + o, dO_b + o, kIdS, kk > 0);
        }
        umma_commit(dp_full);
        if (L::kSharedDQ && n > 0) {
          // The previous dQ tile (in the S^T columns) must have been read out.
          ok = mbar_wait(dq_free, (n - 1) & 1, 45);
          if (!ok) break;
          tc_fence_after();
        }
        // S^T = K Q^T (K = d).
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t o = static_cast<uint64_t>(((kk >> 2) * (128 * 128) + (kk & 3) * 32) >> 4);
          umma_bf16_ss(tmem + L::kColS, dK_a + o, dQ_b + o, kIdS, kk > 0);
        }
        umma_commit(s_full);
        ok = mbar_wait(ds_full, n & 1, 46);
        if (!ok) break;
        tc_fence_after();
        if (!L::kSharedDQ && n > 0) {
          ok = mbar_wait(dq_free, (n - 1) & 1, 47);
          if (!ok) break;
          tc_fence_after();
        }
        // dQ tile = dS K (K = 128 keys) first, so that its read-out overlaps
        // the dV and dK products.
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t o = static_cast<uint64_t>((kk * (16 * 128)) >> 4);
          umma_bf16_ss(tmem + L::kColDQ, dS_a + o, dK_b + o, kIdQ, kk > 0);
        }
        umma_commit(dq_full);
        // dV += P^T dO, dK += dS^T Q (K = 128 query rows; A from TMEM: the 16
        // queries of step kk lie in query half kk / 4, at P^T or dS^T
        // columns 64 (kk / 4) + 32 + 8 (kk % 4), resp. 64 (kk / 4) + 8 (kk % 4)).
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t o = static_cast<uint64_t>((kk * (16 * 128)) >> 4);
          const uint32_t pcol = (kk >> 2) * 64 + 32 + (kk & 3) * 8;
          umma_bf16_ts(tmem + L::kColDV, tmem + L::kColDP + pcol, dO_mn + o, kIdG, (n > 0 || kk > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t o = static_cast<uint64_t>((kk * (16 * 128)) >> 4);
          const uint32_t dcol = (kk >> 2) * 64 + (kk & 3) * 8;
          umma_bf16_ts(tmem + L::kColDK, tmem + L::kColDP + dcol, dQ_mn + o, kIdG, (n > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&q_empty[st]);
      }
      umma_commit(dkv_done);
      mbar_wait(dkv_done, 0, 48);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- key rows, then query rows
    const int quarter = warp & 3;             // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;         // query columns (weights) / head-dim columns (dQ) of this thread
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const int kj = k0 + row;  // this thread's key
    const int c0 = half * 64; // first query column of this thread's half
    const bool issuer = lane == 0 && quarter == 2;  // the first warp of each half issues its dQ reduces
    bool ok = true;
    // A query row's -LSE log2(e) (-inf for a row that saw no key: its weights
    // are 0) and D, read one item ahead by the first half.
    auto row_vals = [&](int n, float& nl2, float& dd) {
      nl2 = -INFINITY;
      dd = 0.f;
      if (n < n_items) {
        const int qi = item_q0(n) + row;
        if (qi < p.Nq) {
          const size_t r = static_cast<size_t>(item_bh(n)) * p.Nq + qi;
          const float l = __ldg(p.lse + r);
          nl2 = l == -INFINITY ? -INFINITY : -l * 1.4426950408889634f;
          dd = __ldg(p.dsum + r);
        }
      }
    };
    float l_next = 0.f, d_next = 0.f;
    if (half == 0) row_vals(0, l_next, d_next);
    const float sl = p.scale_log2;
    for (int n = 0; ok && n < n_items; ++n) {
      const int bh = item_bh(n), q0 = item_q0(n);
      // The item's 128 row values: one per first-half thread into shared
      // memory, then every weight thread reads the 64 of its half.
      float* nls = reinterpret_cast<float*>(smem + L::kRowOff + (n & 1) * L::kRowBytes);
      float* dsum = nls + 128;
      if (half == 0) {
        nls[row] = l_next;
        dsum[row] = d_next;
        mbar_arrive(&rows_ready[n & 1]);
        row_vals(n + 1, l_next, d_next);
      }
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(&rows_ready[n & 1], (n >> 1) & 1, 49));
      if (!ok) break;
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(dp_full, n & 1, 51));
      if (!ok) break;
      tc_fence_after();
      // This half's 64 dP^T columns first: their columns then take dS^T and P^T.
      uint32_t dp[64];
      tmem_ld32(lane_base + L::kColDP + c0, *reinterpret_cast<uint32_t(*)[32]>(dp + 0));
      tmem_ld32(lane_base + L::kColDP + c0 + 32, *reinterpret_cast<uint32_t(*)[32]>(dp + 32));
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(s_full, n & 1, 50));
      if (!ok) break;
      tc_fence_after();
      // Query c of the tile is allowed for this key iff c < Nq - q0, and
      // (causal) kj <= q0 + c + diag; tiles wholly inside skip the test.
      int c_hi = p.Nq - q0;                                     // columns >= c_hi: past Nq
      const int c_lo = p.causal ? kj - diag - q0 : -0x7FFFFFFF;  // columns < c_lo: masked
      if (p.window_left > 0) c_hi = min(c_hi, kj - diag + p.window_left - q0);  // left window
      const bool key_ok = kj < p.Nk;
      const bool masked = !(key_ok && c_lo <= c0 && c_hi >= c0 + 64);
      BwdBiasRow br;
      if constexpr (BIAS) br = bwd_bias_row(p, bh, q0, kj);
      const uint32_t ds_row = sbase + L::kDSOff + half * (128 * 128) + row * 128;
      if (n > 0) {
        // This half's part of the dS region was the staging buffer of its
        // previous dQ chunks: their TMA reduces must have finished reading it.
        const int g1 = n * (D / 64) - 1;  // this half's last staging use of the previous item
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(&red_free[half], g1 & 1, 54));
        if (!ok) break;
      }
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {  // 32 query columns per chunk
        uint32_t sv[32];
        tmem_ld32(lane_base + L::kColS + c0 + ch * 32, sv);
        uint32_t pw[16], dw[16];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const int c = c0 + ch * 32 + e;
          const uint4 nl4 = ld_shared_v4(smem_u32(nls + c));
          const uint4 dd4 = ld_shared_v4(smem_u32(dsum + c));
          const float nl[4] = {__uint_as_float(nl4.x), __uint_as_float(nl4.y), __uint_as_float(nl4.z),
                               __uint_as_float(nl4.w)};
          const float dd[4] = {__uint_as_float(dd4.x), __uint_as_float(dd4.y), __uint_as_float(dd4.z),
                               __uint_as_float(dd4.w)};
#pragma unroll
          for (int u = 0; u < 4; u += 2) {
            float x0, x1, p0, p1, t0, t1, d0, d1;
            ffma2(x0, x1, __uint_as_float(sv[e + u]), __uint_as_float(sv[e + u + 1]), sl, sl, nl[u], nl[u + 1]);
            if constexpr (BIAS) {
              x0 += bwd_bias_at(br, c + u, key_ok, c_lo, c_hi);
              x1 += bwd_bias_at(br, c + u + 1, key_ok, c_lo, c_hi);
            }
            p0 = ex2(x0);
            p1 = ex2(x1);
            if (masked) {
              const int cc = c + u;
              if (!(key_ok && cc < c_hi && cc >= c_lo)) p0 = 0.f;
              if (!(key_ok && cc + 1 < c_hi && cc + 1 >= c_lo)) p1 = 0.f;
            }
            fsub2(t0, t1, __uint_as_float(dp[ch * 32 + e + u]), __uint_as_float(dp[ch * 32 + e + u + 1]), dd[u],
                  dd[u + 1]);
            fmul2(d0, d1, p0, p1, t0, t1);
            pw[(e + u) >> 1] = pack_bf16(p0, p1);
            dw[(e + u) >> 1] = pack_bf16(d0, d1);
          }
        }
        // dS^T and P^T over this half's dP^T columns (the row is in registers).
        tmem_st16(lane_base + L::kColDP + c0 + ch * 16, dw);
        tmem_st16(lane_base + L::kColDP + c0 + 32 + ch * 16, pw);
        // dS^T row into shared memory: 16-byte unit uu of this half's 64-query
        // box at position uu ^ (row & 7) (128-byte swizzle).
#pragma unroll
        for (int u4 = 0; u4 < 4; ++u4) {
          const int uu = ch * 4 + u4;
          st_shared_v4(ds_row + ((uu ^ (row & 7)) << 4), dw[4 * u4], dw[4 * u4 + 1], dw[4 * u4 + 2], dw[4 * u4 + 3]);
        }
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_full);

      // dQ tile rows (TMEM lane = query row), this half's D/2 columns: scale
      // and add into the accumulator.
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(dq_full, n & 1, 52));
      if (!ok) break;
      tc_fence_after();
      // 32 columns at a time: scale, stage as [128 rows][32] f32 (128-byte
      // swizzle, conflict-free row writes) in this half's 16 KB buffer of the
      // dS region (free: the dQ product has read dS), and the half's issuing
      // thread adds the chunk into the f32 accumulator with a TMA reduce.
      constexpr int kCh = D / 64;  // chunks per half
#pragma unroll 1
      for (int ch = 0; ok && ch < kCh; ++ch) {
        const int g = n * kCh + ch;  // this half's running staging use
        uint32_t v[32];
        tmem_ld32(lane_base + L::kColDQ + half * (D / 2) + ch * 32, v);
        if (ch == kCh - 1) {
          // This thread's part of the dQ tile is in registers: once every
          // weight warp got here, the next dQ product may start.
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(dq_free);
        }
        if (ch > 0) {
          // The previous chunk of this item used the same buffer.
          ok = __all_sync(0xFFFFFFFFu, mbar_wait(&red_free[half], (g - 1) & 1, 56));
          if (!ok) break;
        }
        const uint32_t stg = sbase + L::kDSOff + half * (128 * 128) + row * 128;
#pragma unroll
        for (int k = 0; k < 8; ++k)
          st_shared_v4(stg + ((k ^ (row & 7)) << 4), __float_as_uint(__uint_as_float(v[4 * k]) * p.scale),
                       __float_as_uint(__uint_as_float(v[4 * k + 1]) * p.scale),
                       __float_as_uint(__uint_as_float(v[4 * k + 2]) * p.scale),
                       __float_as_uint(__uint_as_float(v[4 * k + 3]) * p.scale));
        fence_proxy_async_smem();
        mbar_arrive(&red_full[half]);
        if (issuer) {
          if (!mbar_wait(&red_full[half], g & 1, 57)) {
            ok = false;
          } else {
            tma_reduce_add_3d(&tmDQ, smem + L::kDSOff + half * (128 * 128), half * (D / 2) + ch * 32, q0, bh);
            bulk_commit();
            bulk_wait_read<0>();
            mbar_arrive(&red_free[half]);
          }
        }
        ok = __all_sync(0xFFFFFFFFu, ok);
      }
      if (!ok) break;
    }

    // dK, dV rows of this key (zeros when no query row sees the tile), this
    // half's D/2 columns.  The tensor-memory loads are warp-collective: every
    // lane runs them, and only the stores depend on the lane's key being
    // inside Nk.
    if (ok && n_items > 0) {
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(dkv_done, 0, 53));
      if (ok) tc_fence_after();
    }
    if (ok) {
      const bool store = kj < p.Nk;
      const size_t off = (static_cast<size_t>(bkv) * p.Nk + kj) * D;
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        const uint32_t col = which == 0 ? L::kColDK : L::kColDV;
        const float mul = which == 0 ? p.scale : 1.f;
        void* outp = which == 0 ? p.dk : p.dv;
#pragma unroll 1
        for (int ch = half * (D / 64); ch < (half + 1) * (D / 64); ++ch) {
          uint32_t v[32];
          if (n_items > 0) {
            tmem_ld32(lane_base + col + ch * 32, v);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = 0u;
          }
          if (!store) continue;
          if (p.g_f32) {
            float4* o4 = reinterpret_cast<float4*>(static_cast<float*>(outp) + off + ch * 32);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              o4[e] = make_float4(__uint_as_float(v[4 * e]) * mul, __uint_as_float(v[4 * e + 1]) * mul,
                                  __uint_as_float(v[4 * e + 2]) * mul, __uint_as_float(v[4 * e + 3]) * mul);
          } else {
            uint4* o4 = reinterpret_cast<uint4*>(static_cast<uint16_t*>(outp) + off + ch * 32);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int x = 8 * e;
              o4[e] = make_uint4(pack_bf16(__uint_as_float(v[x]) * mul, __uint_as_float(v[x + 1]) * mul),
                                 pack_bf16(__uint_as_float(v[x + 2]) * mul, __uint_as_float(v[x + 3]) * mul),
                                 pack_bf16(__uint_as_float(v[x + 4]) * mul, __uint_as_float(v[x + 5]) * mul),
                                 pack_bf16(__uint_as_float(v[x + 6]) * mul, __uint_as_float(v[x + 7]) * mul));
            }
          }
        }
      }
    }
  }

  // Every dQ reduce of this CTA must have read its staging buffer before the
  // CTA (and its shared memory) ends; the global adds complete with the grid.
  if (warp >= 2 && lane == 0 && (warp & 3) == 2) bulk_wait_read<0>();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace attn
