// Attention backward at head dim 256 (the same products as bwd.cuh: the
// derivative of the forward of "Compilers and Kernels", section
// "FlashAttention changes the algorithm around IO", with the weights
// recomputed from the saved row logsumexp as in the flash-style backward of
// "Tang: a compiler that derives GPU kernels and bounds how fast they can run",
// abstract; head dim 256 is the "derived head-dim-256 attention" there).
//
// At d = 256 the dK and dV accumulators of one 128-key tile alone fill the
// 512 tensor-memory columns, so a key tile is served by two CTAs, one per
// half of the head dim (h = 0, 1): CTA h keeps dK[:, h], dV[:, h] (128 columns
// each) and adds dQ[:, h].  Both recompute the full S^T and dP^T (contraction
// over all 256 columns), which costs 32 of every 56 products of an item twice
// but needs no exchange between the two.  K and V (64 KB each) stay in shared
// memory; items are 64-query tiles (Q and dO 32 KB each, one stage), so the
// score tiles are N = 64 products:
//   S^T  = K Q^T        [128 keys][64 queries]    (tensor memory, 64 columns)
//   dP^T = V dO^T       [128 keys][64 queries]
//   P^T, dS^T as in bf16 over the dP^T columns
//   dV_h += P^T dO_h,  dK_h += dS^T Q_h            (A from tensor memory)
//   dQ^T_h = K_h^T dS^T [128 head-dim rows][64 queries] (dS^T staged in shared
//            memory), added to a transposed f32 accumulator dQacc^T[bh][d][q]
//            by TMA reduce-adds; the post kernel transposes it back.
// Tensor memory: dK_h 128, dV_h 128, S^T 64, dP^T 64, dQ^T 64 columns.
// Roles as in bwd.cuh: warp 0 TMA producer, warp 1 MMA issuer, warps 2..9 two
// per TMEM lane quarter, each thread one key row and 32 of the item's 64 query
// columns (weights), then one head-dim row and 32 query columns (dQ^T).
#pragma once

#include "bwd.cuh"

namespace attn {

struct BwdWideLayout {
  static constexpr int D = 256;
  static constexpr int kThreads = 320;
  static constexpr int kBQ = 64;                       // query rows per item
  static constexpr int kKVTile = 128 * D * 2;          // [128 keys][256] bf16: 4 boxes [128][64] of 16 KB
  static constexpr int kQTile = kBQ * D * 2;           // [64 rows][256] bf16: 4 boxes [64][64] of 8 KB
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kKVTile;
  static constexpr int kQOff = kVOff + kKVTile;
  static constexpr int kDOOff = kQOff + kQTile;
  static constexpr int kDSOff = kDOOff + kQTile;       // dS^T [128 keys][64 queries] bf16 (16 KB), then
                                                       // half 0's dQ^T staging [128][32] f32
  static constexpr int kStgOff = kDSOff + 16384;       // half 1's dQ^T staging [128][32] f32
  static constexpr int kRowOff = kStgOff + 16384;      // 2 x (-LSE log2 e [64], D [64]) f32
  static constexpr int kRowBytes = 2 * kBQ * 4;
  static constexpr int kBarOff = kRowOff + 2 * kRowBytes;
  // kv_full, q_full, q_empty, do_full, do_empty, s_full, dp_full, ds_full, dq_full, dq_free, dkv_done,
  // rows_ready[2], red_full[2], red_free[2]
  static constexpr int kNumBars = 17;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kMiscOff + 16;
  static constexpr int kAlloc = kBytes + 128;          // the base is checked for 1024-byte alignment
  static constexpr int kColDK = 0;
  static constexpr int kColDV = 128;
  static constexpr int kColS = 256;
  static constexpr int kColDP = 320;                   // half h: dS^T in [32h, 32h + 16), P^T in [32h + 16, 32h + 32)
  static constexpr int kColDQ = 384;
  static_assert(kBytes + 128 <= 232448, "shared memory budget");
};

// dq[bh][q][c] = dqT[bh][c][q] (f32 accumulator, rows of ld floats) as bf16 (RNE) or f32;
// one 32 x 32 tile per block of 32 x 8 threads.
__global__ void bwd_post_transpose_kernel(const float* dqT, void* dq, int BH, int Nq, int ld, int d, int g_f32) {
  __shared__ float tile[32][33];
  const int q0 = blockIdx.x * 32, c0 = blockIdx.y * 32;
  for (int bh = blockIdx.z; bh < BH; bh += gridDim.z) {
    const float* src = dqT + static_cast<size_t>(bh) * d * ld;
    for (int r = threadIdx.y; r < 32; r += 8) {
      const int q = q0 + threadIdx.x;
      tile[r][threadIdx.x] = q < Nq ? src[static_cast<size_t>(c0 + r) * ld + q] : 0.f;
    }
    __syncthreads();
    for (int r = threadIdx.y; r < 32; r += 8) {
      const int q = q0 + r;
      if (q >= Nq) continue;
      const size_t off = (static_cast<size_t>(bh) * Nq + q) * d + c0 + threadIdx.x;
      const float v = tile[threadIdx.x][r];
      if (g_f32) {
        static_cast<float*>(dq)[off] = v;
      } else {
        static_cast<uint16_t*>(dq)[off] = static_cast<uint16_t>(pack_bf16(v, 0.f) & 0xFFFFu);
      }
    }
    __syncthreads();
  }
}

template <bool BIAS>
__global__ void __launch_bounds__(320, 1)
    attn_bwd_wide_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                         const __grid_constant__ CUtensorMap tmDQT, const BwdParams p) {
  using L = BwdWideLayout;
  constexpr int D = L::D;
  constexpr int BQ = L::kBQ;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  if (pad + L::kBytes > static_cast<uint32_t>(L::kAlloc)) {
    if (threadIdx.x == 0) report_error(5 /* ATTN_ERR_LAUNCH */, 31, static_cast<int>(pad));
    return;
  }
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw + pad;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* kv_full = bars;
  uint64_t* q_full = bars + 1;
  uint64_t* q_empty = bars + 2;
  uint64_t* do_full = bars + 3;
  uint64_t* do_empty = bars + 4;
  uint64_t* s_full = bars + 5;
  uint64_t* dp_full = bars + 6;
  uint64_t* ds_full = bars + 7;
  uint64_t* dq_full = bars + 8;
  uint64_t* dq_free = bars + 9;
  uint64_t* dkv_done = bars + 10;
  uint64_t* rows_ready = bars + 11;  // [2]
  uint64_t* red_full = bars + 13;    // [2] a half's [128][32] f32 dQ^T chunk is staged
  uint64_t* red_free = bars + 15;    // [2] its TMA reduce has finished reading the staging buffer
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int BHkv = p.B * p.Hkv;
  const int h = static_cast<int>(blockIdx.x & 1u);         // head-dim half of dK, dV, dQ
  const int kt = static_cast<int>(blockIdx.x >> 1) / BHkv;  // key tile 0 first (seen by the most rows)
  const int bkv = static_cast<int>(blockIdx.x >> 1) - kt * BHkv;
  const int b = bkv / p.Hkv;
  const int kvh = bkv - b * p.Hkv;
  const int k0 = kt * 128;
  const int G = p.Hq / p.Hkv;
  const int diag = p.Nk - p.Nq;
  int qt_lo, qt_hi;
  bwd_query_tiles(p, k0, BQ, qt_lo, qt_hi);
  const int per_head = qt_hi - qt_lo;
  const int n_items = G * per_head;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    mbar_init(do_full, 1);
    mbar_init(do_empty, 1);
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(ds_full, 8);
    mbar_init(dq_full, 1);
    mbar_init(dq_free, 8);
    mbar_init(dkv_done, 1);
    mbar_init(&rows_ready[0], BQ);
    mbar_init(&rows_ready[1], BQ);
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

  auto item_bh = [&](int n) { return b * p.Hq + kvh * G + n / per_head; };
  auto item_q0 = [&](int n) { return (qt_lo + n % per_head) * BQ; };

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0 && n_items > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
      mbar_expect_tx(kv_full, 2 * L::kKVTile);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        tma_load_3d(smem + L::kKOff + c * (128 * 128), &tmK, kv_full, c * 64, k0, bkv);
        tma_load_3d(smem + L::kVOff + c * (128 * 128), &tmV, kv_full, c * 64, k0, bkv);
      }
      int n_do = 0, n_q = 0;  // loads issued
      for (int n = 0; n < n_items; ++n) {
        const int bh = item_bh(n), q0 = item_q0(n);
        // dO first: the item's first product (dP^T) reads it, and its slot
        // frees after the previous item's dV product, before Q's (dK).
        if (!mbar_wait(do_empty, (n & 1) ^ 1, 70)) break;
        mbar_expect_tx(do_full, L::kQTile);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + L::kDOOff + c * (BQ * 128), &tmDO, do_full, c * 64, q0, bh);
        n_do = n + 1;
        if (!mbar_wait(q_empty, (n & 1) ^ 1, 71)) break;
        mbar_expect_tx(q_full, L::kQTile);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + L::kQOff + c * (BQ * 128), &tmQ, q_full, c * 64, q0, bh);
        n_q = n + 1;
      }
      // Drain: never leave the CTA with a copy still writing shared memory.
      // One stage each: a load is issued only after the previous one was
      // consumed, so only the last of each can still be in flight.
      mbar_wait(kv_full, 0, 72);
      if (n_do > 0) mbar_wait(do_full, (n_do - 1) & 1, 73);
      if (n_q > 0) mbar_wait(q_full, (n_q - 1) & 1, 74);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0 && n_items > 0) {
      constexpr uint32_t kIdS = idesc_bf16_f32(128, BQ, 0, 0);   // S^T, dP^T: K-major A and B, N = 64
      constexpr uint32_t kIdG = idesc_bf16_f32(128, 128, 0, 1);  // dV_h, dK_h: A from TMEM, B MN-major
      constexpr uint32_t kIdQ = idesc_bf16_f32(128, BQ, 1, 1);   // dQ^T_h: A (K_h^T), B (dS^T) MN-major
      const uint64_t dK_a = sdesc_sw128(sbase + L::kKOff, 16, 1024);
      const uint64_t dV_a = sdesc_sw128(sbase + L::kVOff, 16, 1024);
      const uint64_t dQ_b = sdesc_sw128(sbase + L::kQOff, 16, 1024);
      const uint64_t dO_b = sdesc_sw128(sbase + L::kDOOff, 16, 1024);
      // Head-dim half h: boxes 2h, 2h + 1 of K (16 KB apart) and of Q, dO (8 KB apart).
      const uint64_t dKh_mn = sdesc_sw128(sbase + L::kKOff + h * 2 * (128 * 128), 128 * 128, 1024);
      const uint64_t dQh_mn = sdesc_sw128(sbase + L::kQOff + h * 2 * (BQ * 128), BQ * 128, 1024);
      const uint64_t dOh_mn = sdesc_sw128(sbase + L::kDOOff + h * 2 * (BQ * 128), BQ * 128, 1024);
      const uint64_t dS_mn = sdesc_sw128(sbase + L::kDSOff, BQ * 128, 1024);
      bool ok = mbar_wait(kv_full, 0, 75);
      if (ok) tc_fence_after();
      for (int n = 0; ok && n < n_items; ++n) {
        // dP^T = V dO^T (K = 256): its slot is free once the previous item's
        // dV and dK products (issued earlier) have read P^T and dS^T from it.
        ok = mbar_wait(do_full, n & 1, 76);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t oa = static_cast<uint64_t>(((kk >> 2) * (128 * 128) + (kk & 3) * 32) >> 4);
          const uint64_t ob = static_cast<uint64_t>(((kk >> 2) * (BQ * 128) + (kk & 3) * 32) >> 4);
          umma_bf16_ss(tmem + L::kColDP, dV_a + oa, dO_b + ob, kIdS, kk > 0);
        }
        umma_commit(dp_full);
        // S^T = K Q^T (K = 256): the previous item's weights read S^T before
        // they signalled ds_full, which this thread waited for.
        ok = mbar_wait(q_full, n & 1, 77);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t oa = static_cast<uint64_t>(((kk >> 2) * (128 * 128) + (kk & 3) * 32) >> 4);
          const uint64_t ob = static_cast<uint64_t>(((kk >> 2) * (BQ * 128) + (kk & 3) * 32) >> 4);
          umma_bf16_ss(tmem + L::kColS, dK_a + oa, dQ_b + ob, kIdS, kk > 0);
        }
        umma_commit(s_full);
        ok = mbar_wait(ds_full, n & 1, 78);
        if (!ok) break;
        tc_fence_after();
        if (n > 0) {
          // The previous dQ^T tile must have been read out of its columns.
          ok = mbar_wait(dq_free, (n - 1) & 1, 79);
          if (!ok) break;
          tc_fence_after();
        }
        // dQ^T_h = K_h^T dS^T (K = 128 keys) first, so that its read-out
        // overlaps the dV and dK products.
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t o = static_cast<uint64_t>((kk * (16 * 128)) >> 4);
          umma_bf16_ss(tmem + L::kColDQ, dKh_mn + o, dS_mn + o, kIdQ, kk > 0);
        }
        umma_commit(dq_full);
        // dV_h += P^T dO_h, dK_h += dS^T Q_h (K = 64 queries; the 16 queries
        // of step kk lie in query half kk / 2: P^T at columns 32 (kk / 2) + 16
        // + 8 (kk % 2), dS^T at 32 (kk / 2) + 8 (kk % 2)).
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk) {
          const uint64_t o = static_cast<uint64_t>((kk * (16 * 128)) >> 4);
          const uint32_t pcol = (kk >> 1) * 32 + 16 + (kk & 1) * 8;
          umma_bf16_ts(tmem + L::kColDV, tmem + L::kColDP + pcol, dOh_mn + o, kIdG, (n > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(do_empty);
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk) {
          const uint64_t o = static_cast<uint64_t>((kk * (16 * 128)) >> 4);
          const uint32_t dcol = (kk >> 1) * 32 + (kk & 1) * 8;
          umma_bf16_ts(tmem + L::kColDK, tmem + L::kColDP + dcol, dQh_mn + o, kIdG, (n > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(q_empty);
      }
      umma_commit(dkv_done);
      mbar_wait(dkv_done, 0, 80);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- key rows, then head-dim rows
    const int quarter = warp & 3;             // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;         // query columns [32 half, 32 half + 32) of the item
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const int kj = k0 + row;                  // this thread's key (weights)
    const int c0 = half * 32;
    const bool row_writer = half == 0 && row < BQ;
    const bool issuer = lane == 0 && quarter == 2;  // the first warp of each half issues its dQ^T reduce
    bool ok = true;
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
    if (row_writer) row_vals(0, l_next, d_next);
    const float sl = p.scale_log2;
    for (int n = 0; ok && n < n_items; ++n) {
      const int bh = item_bh(n), q0 = item_q0(n);
      float* nls = reinterpret_cast<float*>(smem + L::kRowOff + (n & 1) * L::kRowBytes);
      float* dsum = nls + BQ;
      if (row_writer) {
        nls[row] = l_next;
        dsum[row] = d_next;
        mbar_arrive(&rows_ready[n & 1]);
        row_vals(n + 1, l_next, d_next);
      }
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(&rows_ready[n & 1], (n >> 1) & 1, 81));
      if (!ok) break;
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(dp_full, n & 1, 82));
      if (!ok) break;
      tc_fence_after();
      uint32_t dp[32];
      tmem_ld32(lane_base + L::kColDP + c0, dp);
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(s_full, n & 1, 83));
      if (!ok) break;
      tc_fence_after();
      uint32_t sv[32];
      tmem_ld32(lane_base + L::kColS + c0, sv);
      if (n > 0) {
        // The dS^T region was half 0's staging buffer for the previous item:
        // its TMA reduce must have finished reading it.
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(&red_free[0], (n - 1) & 1, 84));
        if (!ok) break;
      }
      int c_hi = p.Nq - q0;
      const int c_lo = p.causal ? kj - diag - q0 : -0x7FFFFFFF;
      if (BIAS && p.window_left > 0) c_hi = min(c_hi, kj - diag + p.window_left - q0);  // left window
      const bool key_ok = kj < p.Nk;
      const bool masked = !(key_ok && c_lo <= c0 && c_hi >= c0 + 32);
      BwdBiasRow br;
      if constexpr (BIAS) br = bwd_bias_row(p, bh, q0, kj);
      uint32_t pw[16], dw[16];
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        const int c = c0 + e;
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
          fsub2(t0, t1, __uint_as_float(dp[e + u]), __uint_as_float(dp[e + u + 1]), dd[u], dd[u + 1]);
          fmul2(d0, d1, p0, p1, t0, t1);
          pw[(e + u) >> 1] = pack_bf16(p0, p1);
          dw[(e + u) >> 1] = pack_bf16(d0, d1);
        }
      }
      // dS^T and P^T over this half's dP^T columns, dS^T into shared memory
      // (row `row`, 16-byte units 4 half .. 4 half + 3 in the 128-byte swizzle).
      tmem_st16(lane_base + L::kColDP + c0, dw);
      tmem_st16(lane_base + L::kColDP + c0 + 16, pw);
      const uint32_t ds_row = sbase + L::kDSOff + row * 128;
#pragma unroll
      for (int u4 = 0; u4 < 4; ++u4) {
        const int uu = half * 4 + u4;
        st_shared_v4(ds_row + ((uu ^ (row & 7)) << 4), dw[4 * u4], dw[4 * u4 + 1], dw[4 * u4 + 2], dw[4 * u4 + 3]);
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_full);

      // dQ^T rows (TMEM lane = head-dim row of half h), this thread's 32
      // query columns: scale, stage [128 rows][32] f32 (128-byte swizzle),
      // and the half's issuing thread adds the chunk with a TMA reduce.
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(dq_full, n & 1, 85));
      if (!ok) break;
      tc_fence_after();
      uint32_t v[32];
      tmem_ld32(lane_base + L::kColDQ + c0, v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dq_free);
      if (half == 1 && n > 0) {
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(&red_free[1], (n - 1) & 1, 86));
        if (!ok) break;
      }
      const uint32_t stg_base = half == 0 ? L::kDSOff : L::kStgOff;
      const uint32_t stg = sbase + stg_base + row * 128;
#pragma unroll
      for (int k = 0; k < 8; ++k)
        st_shared_v4(stg + ((k ^ (row & 7)) << 4), __float_as_uint(__uint_as_float(v[4 * k]) * p.scale),
                     __float_as_uint(__uint_as_float(v[4 * k + 1]) * p.scale),
                     __float_as_uint(__uint_as_float(v[4 * k + 2]) * p.scale),
                     __float_as_uint(__uint_as_float(v[4 * k + 3]) * p.scale));
      fence_proxy_async_smem();
      mbar_arrive(&red_full[half]);
      if (issuer) {
        if (!mbar_wait(&red_full[half], n & 1, 87)) {
          ok = false;
        } else {
          tma_reduce_add_3d(&tmDQT, smem + stg_base, q0 + c0, h * 128, bh);
          bulk_commit();
          bulk_wait_read<0>();
          mbar_arrive(&red_free[half]);
        }
      }
      ok = __all_sync(0xFFFFFFFFu, ok);
    }

    // dK_h, dV_h rows of this key (zeros when no query row sees the tile):
    // this thread's 64 of the CTA's 128 head-dim columns.  The tensor-memory
    // loads run on every lane; only the stores depend on the key being < Nk.
    if (ok && n_items > 0) {
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(dkv_done, 0, 88));
      if (ok) tc_fence_after();
    }
    if (ok) {
      const bool store = kj < p.Nk;
      const size_t off = (static_cast<size_t>(bkv) * p.Nk + kj) * D + h * 128;
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        const uint32_t col = which == 0 ? L::kColDK : L::kColDV;
        const float mul = which == 0 ? p.scale : 1.f;
        void* outp = which == 0 ? p.dk : p.dv;
#pragma unroll 1
        for (int ch = half * 2; ch < half * 2 + 2; ++ch) {
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

  // Every dQ^T reduce of this CTA must have completed before it exits.
  if (warp >= 2 && lane == 0 && (warp & 3) == 2) bulk_wait_all();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace attn
