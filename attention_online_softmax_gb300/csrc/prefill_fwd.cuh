// Fused attention forward (prefill) for sm_103a.
//
// One CTA computes one 128-row query tile of one (batch, query head) against
// the key/value tiles that row block may see, following the block recurrence
// of "Compilers and Kernels", section "FlashAttention changes the algorithm
// around IO": for each key block B_t the row state (m, l, o) is updated by
//     m_t = max(m_{t-1}, b_t),  alpha_t = exp(m_{t-1} - m_t),
//     l_t = alpha_t l_{t-1} + sum exp(S - m_t),  o_t = alpha_t o_{t-1} + sum exp(S - m_t) v,
// and O = o_T / l_T, LSE = m_T + ln l_T at the end.  Scores never leave the SM.
//
// Roles (192 threads):
//   warp 0      TMA producer: Q once, then K_t, V_t tiles into a STAGES-deep
//               shared-memory ring (128-byte swizzle), gated by mbarriers.
//   warp 1      allocates tensor memory; one thread issues tcgen05.mma:
//               S_t = Q K_t^T into one of two TMEM score buffers, and
//               O += P_t V_t into the TMEM accumulator.
//   warps 2..5  softmax warpgroup, one thread per query row: reads S_t from
//               TMEM, applies scale*log2(e) and the causal/ragged mask,
//               updates the running max, writes P_t = 2^(x - m) as bf16 into
//               shared memory (A operand of the second MMA), rescales O in
//               TMEM when the max moved, and finally writes O / l and LSE.
//
// Work is done in base 2: x = s * scale * log2(e), p = 2^(x - m), and
// LSE = (m + log2 l) * ln 2.  The reference max m is only moved when a tile's
// max exceeds it by more than kRescaleLog2 (2^8): the result is exact for any
// reference value (numerator and denominator share it) and the bound keeps
// every p <= 256, so most tiles skip the O rescale.
#pragma once

#include "ptx.cuh"

namespace attn {

constexpr int kBM = 128;                 // query rows per CTA (TMEM lanes)
constexpr float kRescaleLog2 = 8.0f;
constexpr int kPrefillThreads = 192;

struct PrefillParams {
  void* o;
  float* lse;
  int B, Hq, Hkv, Nq, Nk;
  int causal;
  int o_f32;
  int n_qtiles;
  float scale_log2;  // scale * log2(e)
};

template <int D, int BN, int STAGES>
struct PrefillLayout {
  static constexpr int kQBytes = kBM * D * 2;
  static constexpr int kKVBytes = BN * D * 2;
  static constexpr int kPBytes = kBM * BN * 2;
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = kQOff + kQBytes;
  static constexpr int kPOff = kKVOff + STAGES * kKVBytes;
  static constexpr int kBarOff = kPOff + kPBytes;
  // q_full, kv_full[S], kv_empty[S], s_full[2], s_free[2], p_full, pv_done, mma_drain
  static constexpr int kNumBars = 1 + 2 * STAGES + 7;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kMiscOff + 16;
  static constexpr int kAlloc = kBytes + 1024;  // room to align the dynamic base to 1024
  static constexpr int kTmemCols = 512;
  static_assert(D + 2 * BN <= kTmemCols, "tensor memory budget");
  static_assert(kBytes + 1024 <= 232448, "shared memory budget");
  static_assert(D % 64 == 0 && BN % 64 == 0, "tile shapes");
};

template <int D, int BN, int STAGES>
__global__ void __launch_bounds__(kPrefillThreads, 1)
    prefill_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
  using L = PrefillLayout<D, BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const uint32_t sbase = smem_u32(smem);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = bars + 1 + STAGES;
  uint64_t* s_full = bars + 1 + 2 * STAGES;
  uint64_t* s_free = s_full + 2;
  uint64_t* p_full = s_free + 2;
  uint64_t* pv_done = p_full + 1;
  uint64_t* mma_drain = pv_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Flat grid: block = bh * n_qtiles + i, with the query tiles of one head
  // visited longest (causal) first.
  const int bh = static_cast<int>(blockIdx.x) / p.n_qtiles;
  const int qt = p.n_qtiles - 1 - (static_cast<int>(blockIdx.x) - bh * p.n_qtiles);
  if (bh >= p.B * p.Hq || qt < 0) return;  // never taken with the host's grid
  const int b = bh / p.Hq;
  const int h = bh - b * p.Hq;
  const int kvh = b * p.Hkv + h / (p.Hq / p.Hkv);
  const int q0 = qt * kBM;
  const int diag = p.Nk - p.Nq;  // key j allowed for row i iff j <= i + diag (causal)

  int kend = p.Nk;
  if (p.causal) {
    const int last_row = min(q0 + kBM, p.Nq) - 1;
    kend = min(p.Nk, last_row + diag + 1);
  }
  const int n_tiles = kend > 0 ? (kend + BN - 1) / BN : 0;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 4);
    }
    mbar_init(p_full, 4);
    mbar_init(pv_done, 1);
    mbar_init(mma_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0 && n_tiles > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_expect_tx(q_full, L::kQBytes);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tma_load_3d(smem + L::kQOff + c * (kBM * 128), &tmQ, q_full, c * 64, q0, bh);
      int issued = 0;
      for (int item = 0; item < 2 * n_tiles; ++item) {
        const int st = item % STAGES;
        const uint32_t ph = (item / STAGES) & 1;
        if (*abort_flag || !mbar_wait(&kv_empty[st], ph ^ 1, 1)) {
          *abort_flag = 1;
          break;
        }
        mbar_expect_tx(&kv_full[st], L::kKVBytes);
        const CUtensorMap* map = (item & 1) ? &tmV : &tmK;
        const int krow = (item >> 1) * BN;
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + L::kKVOff + st * L::kKVBytes + c * (BN * 128), map, &kv_full[st], c * 64, krow,
                      kvh);
        issued = item + 1;
      }
      // Drain: never leave the CTA with a copy still writing shared memory.
      mbar_wait(q_full, 0, 2);
      for (int item = max(0, issued - STAGES); item < issued; ++item)
        mbar_wait(&kv_full[item % STAGES], (item / STAGES) & 1, 3);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0 && n_tiles > 0) {
      constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, BN, 0, 0);  // Q K-major, K K-major
      constexpr uint32_t kIdescO = idesc_bf16_f32(kBM, D, 0, 1);   // P K-major, V MN-major
      const uint32_t tm_o = tmem;
      bool ok = mbar_wait(q_full, 0, 10);
      for (int t = 0; ok && t <= n_tiles; ++t) {
        if (t < n_tiles) {
          const int item = 2 * t;
          const int st = item % STAGES;
          ok = mbar_wait(&s_free[t & 1], ((t >> 1) & 1) ^ 1, 11) && mbar_wait(&kv_full[st], (item / STAGES) & 1, 12);
          if (!ok) break;
          tc_fence_after();
          const uint32_t tm_s = tmem + D + (t & 1) * BN;
          const uint32_t sq = sbase + L::kQOff;
          const uint32_t sk = sbase + L::kKVOff + st * L::kKVBytes;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t da = sdesc_sw128(sq + (kk >> 2) * (kBM * 128) + (kk & 3) * 32, 16, 1024);
            const uint64_t db = sdesc_sw128(sk + (kk >> 2) * (BN * 128) + (kk & 3) * 32, 16, 1024);
            umma_bf16_ss(tm_s, da, db, kIdescS, kk > 0);
          }
          umma_commit(&kv_empty[st]);
          umma_commit(&s_full[t & 1]);
        }
        if (t > 0) {
          const int j = t - 1;
          const int item = 2 * j + 1;
          const int st = item % STAGES;
          ok = mbar_wait(p_full, j & 1, 13) && mbar_wait(&kv_full[st], (item / STAGES) & 1, 14);
          if (!ok) break;
          tc_fence_after();
          const uint32_t sp = sbase + L::kPOff;
          const uint32_t sv = sbase + L::kKVOff + st * L::kKVBytes;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint64_t da = sdesc_sw128(sp + (kk >> 2) * (kBM * 128) + (kk & 3) * 32, 16, 1024);
            const uint64_t db = sdesc_sw128(sv + kk * (16 * 128), BN * 128, 1024);
            umma_bf16_ss(tm_o, da, db, kIdescO, (j > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&kv_empty[st]);
          umma_commit(pv_done);
        }
      }
      if (!ok) *abort_flag = 1;
      // Every MMA this thread issued must be complete before TMEM is freed.
      umma_commit(mma_drain);
      mbar_wait(mma_drain, 0, 15);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- softmax warpgroup
    const int quarter = warp & 3;                 // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;          // row within the tile
    const int qrow = q0 + row;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float sl = p.scale_log2;
    // l sums the exact weights (for LSE); lr sums the bf16-rounded weights the
    // P V product uses, so O = o / lr is an exact convex combination of V rows
    // before output rounding.
    float m_ref = -INFINITY;
    float l = 0.f;
    float lr = 0.f;
    bool ok = true;

    for (int t = 0; t < n_tiles; ++t) {
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(&s_full[t & 1], (t >> 1) & 1, 20));
      if (!ok) break;
      tc_fence_after();
      float x[BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(lane_base + D + (t & 1) * BN + c * 32, r);
#pragma unroll
        for (int i = 0; i < 32; ++i) x[c * 32 + i] = __uint_as_float(r[i]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[t & 1]);

      const int k0 = t * BN;
      const bool need_mask = (k0 + BN > p.Nk) || (p.causal && (k0 + BN - 1 > q0 + diag));
      // Eight independent max chains keep the reduction off the critical path.
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
      if (need_mask) {
        const int lim = p.causal ? min(p.Nk - 1, qrow + diag) - k0 : p.Nk - 1 - k0;
#pragma unroll
        for (int j = 0; j < BN; ++j) {
          x[j] = (j <= lim) ? x[j] * sl : -INFINITY;
          mx[j & 7] = fmaxf(mx[j & 7], x[j]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < BN; ++j) {
          x[j] *= sl;
          mx[j & 7] = fmaxf(mx[j & 7], x[j]);
        }
      }
      const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                             fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      const float m_new = fmaxf(m_ref, mt);
      const bool rescale = m_new > m_ref + kRescaleLog2;
      float alpha = 1.f;
      if (rescale) {
        alpha = ex2(m_ref - m_new);  // 0 when m_ref = -inf
        m_ref = m_new;
        l *= alpha;
        lr *= alpha;
      }
      const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
      uint32_t pk[BN / 2];
      float re[2] = {0.f, 0.f};
      float rr[2] = {0.f, 0.f};
#pragma unroll
      for (int j = 0; j < BN; j += 2) {
        const float p0 = ex2(x[j] - m_use);
        const float p1 = ex2(x[j + 1] - m_use);
        const uint32_t w = pack_bf16(p0, p1);
        pk[j / 2] = w;
        re[(j >> 1) & 1] += p0 + p1;
        rr[(j >> 1) & 1] += bf16lo(w) + bf16hi(w);
      }
      l += re[0] + re[1];
      lr += rr[0] + rr[1];

      if (t > 0) {
        // P buffer and O are busy until the previous P V product is complete.
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(pv_done, (t - 1) & 1, 21));
        if (!ok) break;
        tc_fence_after();
        if (__any_sync(0xFFFFFFFFu, rescale)) {
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(lane_base + c * 32, r);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tmem_st32(lane_base + c * 32, r);
          }
          tmem_st_wait();
        }
      }
      // P row -> shared memory, K-major with the 128-byte swizzle.
      const uint32_t prow = sbase + L::kPOff + row * 128;
#pragma unroll
      for (int ch = 0; ch < BN / 8; ++ch) {
        const uint32_t addr = prow + (ch >> 3) * (kBM * 128) + (((ch & 7) ^ (row & 7)) << 4);
        st_shared_v4(addr, pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }

    if (ok && n_tiles > 0) {
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(pv_done, (n_tiles - 1) & 1, 22));
      if (ok) tc_fence_after();
    }
    if (!ok) *abort_flag = 1;
    // Every lane runs the (warp-collective) TMEM loads; only rows < Nq store.
    const bool store = qrow < p.Nq;
    if (ok) {
      const float inv = (lr > 0.f) ? 1.f / lr : 0.f;
      const size_t row_off = (static_cast<size_t>(bh) * p.Nq + qrow) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        if (n_tiles > 0) {
          tmem_ld32(lane_base + c * 32, r);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = 0u;
        }
        if (!store) continue;
        if (p.o_f32) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + row_off + c * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(__uint_as_float(r[4 * i]) * inv, __uint_as_float(r[4 * i + 1]) * inv,
                                 __uint_as_float(r[4 * i + 2]) * inv, __uint_as_float(r[4 * i + 3]) * inv);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + row_off + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int e = 8 * i;
            dst[i] = make_uint4(pack_bf16(__uint_as_float(r[e]) * inv, __uint_as_float(r[e + 1]) * inv),
                                pack_bf16(__uint_as_float(r[e + 2]) * inv, __uint_as_float(r[e + 3]) * inv),
                                pack_bf16(__uint_as_float(r[e + 4]) * inv, __uint_as_float(r[e + 5]) * inv),
                                pack_bf16(__uint_as_float(r[e + 6]) * inv, __uint_as_float(r[e + 7]) * inv));
          }
        }
      }
      if (store)
        p.lse[static_cast<size_t>(bh) * p.Nq + qrow] =
            (l > 0.f) ? (m_ref + lg2(l)) * 0.69314718055994531f : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

}  // namespace attn
