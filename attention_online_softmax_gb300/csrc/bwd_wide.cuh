// Attention backward at head dims 128 and 256 (the same products as bwd.cuh,
// which serves d = 64: the derivative of the forward of "Compilers and
// Kernels", section "FlashAttention changes the algorithm around IO", with the
// weights recomputed from the saved row logsumexp as in the flash-style
// backward of "Tang: a compiler that derives GPU kernels and bounds how fast
// they can run", abstract; head dim 256 is the "derived head-dim-256
// attention" there).
//
// One CTA keeps a 128-key tile's K and V in shared memory and its dK, dV
// accumulators (128 head-dim columns each) in tensor memory, and walks every
// (query head of the group, 64-row query tile) whose rows see its keys.  At
// d = 256 the two accumulators of a key tile alone would fill the 512
// tensor-memory columns, so the tile is served by two CTAs, one per half of
// the head dim (h = 0, 1): CTA h keeps dK[:, h], dV[:, h] and adds dQ[:, h].
// Both recompute the full S^T and dP^T (contraction over all 256 columns),
// which costs 32 of every 56 products of an item twice but needs no exchange
// between the two.  Per item (score tiles are N = 64 products):
//   S^T  = K Q^T        [128 keys][64 queries]
//   dP^T = V dO^T       [128 keys][64 queries]
//   P^T, dS^T as bf16 over the dP^T columns
//   dV_h += P^T dO_h,  dK_h += dS^T Q_h            (A from tensor memory)
//   dQ^T_h = K_h^T dS^T [128 head-dim rows][64 queries] (dS^T staged in shared
//            memory), staged back as [query][head dim] and added to the f32
//            dQ accumulator [bh][q][d] by TMA reduce-adds.
// Tensor memory: dK_h 128, dV_h 128, and two slots of S^T (then dQ^T) and dP^T
// (then P^T, dS^T), 64 columns each: the next item's score products run while
// the weight warps work on the current item.
// Roles: warp 0 TMA producer; warp 1 issues the score products and warp 14
// the gradient products (one thread each); warps 2..9, two per TMEM lane
// quarter, compute the weights (each thread one key row and 32 of the item's
// 64 query columns); warps 10..13, one per lane quarter, read dQ^T out (each
// thread one head-dim row) and add it with TMA reduce-adds, so the weights of
// one item and the read-out of the previous one run side by side.
#pragma once

#include "bwd.cuh"

namespace attn {

template <int D, int STAGES>
struct BwdWideLayout {
  static_assert(D == 128 || D == 256, "head dims of the 64-query-item backward");
  static constexpr int kSplit = D / 128;               // CTAs per key tile (head-dim halves at D = 256)
  static constexpr int kThreads = 480;
  static constexpr int kBQ = 64;                       // query rows per item
  static constexpr int kKVTile = 128 * D * 2;          // [128 keys][D] bf16: D/64 boxes [128][64] of 16 KB
  static constexpr int kQTile = kBQ * D * 2;           // [64 rows][D] bf16: D/64 boxes [64][64] of 8 KB
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kKVTile;
  static constexpr int kQOff = kVOff + kKVTile;        // STAGES x (Q tile, dO tile)
  static constexpr int kStage = 2 * kQTile;
  static constexpr int kDSOff = kQOff + STAGES * kStage;  // dS^T [128 keys][64 queries] bf16 (16 KB)
  // dQ staging, [32 queries][128 head-dim columns] f32 chunks: two buffers at
  // D = 128, one at D = 256 (no room for a second).
  static constexpr int kNumStg = D == 128 ? 2 : 1;
  static constexpr int kStgOff = kDSOff + 16384;
  static constexpr int kRowOff = kStgOff + kNumStg * 16384;  // 2 x (-LSE log2 e [64], D [64]) f32
  static constexpr int kRowBytes = 2 * kBQ * 4;
  static constexpr int kBarOff = kRowOff + 2 * kRowBytes;
  // Barriers: kv_full, stage_full[S], stage_empty[S], q_full[S], q_empty[S],
  // scores_full[2] (S^T and dP^T of a slot), ds_full, dq_full, dq_free[2]
  // (per slot), dkv_done, sc_done, rows_ready[2], red_full[2], red_free[2]
  // (per staging buffer), wo_full[2] (dV, dK staged for their TMA stores)
  // and dv_done (the last dV product has completed).  With two or more stages an item's Q
  // and dO share stage_full / stage_empty; with one stage (D = 256) dO uses
  // those and Q its own pair, so that dO, which the item's first product
  // reads and whose last reader (dV) finishes first, moves on its own.
  static constexpr bool kSplitOps = STAGES == 1;
  static constexpr int kNumBars = 1 + 4 * STAGES + 2 + 6 + 6 + 3;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kMiscOff + 16;
  static constexpr int kAlloc = kBytes + 128;          // the base is checked for 1024-byte alignment
  // Tensor memory: dK_h, dV_h, then two slots (items alternate) of S^T
  // (64 columns; after the weights have read it, the item's dQ^T) and of
  // dP^T (64 columns; query half h's dS^T in [32h, 32h + 16) and P^T in
  // [32h + 16, 32h + 32) once read).
  static constexpr int kColDK = 0;
  static constexpr int kColDV = 128;
  static constexpr int kColS = 256;                    // slot b at kColS + 64 b
  static constexpr int kColDP = 384;                   // slot b at kColDP + 64 b
  static_assert(kBytes + 128 <= 232448, "shared memory budget");
};

template <int D, int STAGES, bool BIAS>
__global__ void __launch_bounds__(480, 1)
    attn_bwd_wide_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                         const __grid_constant__ CUtensorMap tmDQ, const __grid_constant__ CUtensorMap tmDKo,
                         const __grid_constant__ CUtensorMap tmDVo, const BwdParams p) {
  using L = BwdWideLayout<D, STAGES>;
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
  uint64_t* stage_full = bars + 1;                // [STAGES] an item's Q and dO have landed
  uint64_t* stage_empty = stage_full + STAGES;    // [STAGES] its dK product (the last reader) is done
  uint64_t* q_full = stage_empty + STAGES;        // [STAGES] Q has landed (one stage only)
  uint64_t* q_empty = q_full + STAGES;            // [STAGES] its dK product is done (one stage only)
  uint64_t* scores_full = q_empty + STAGES;       // [2] per slot: S^T and dP^T are in tensor memory
  uint64_t* ds_full = scores_full + 2;
  uint64_t* dq_full = ds_full + 1;
  uint64_t* dq_free = dq_full + 1;      // [2] per slot: its dQ^T has been read out
  uint64_t* dkv_done = dq_free + 2;
  uint64_t* sc_done = dkv_done + 1;     // the score issuer's products have completed
  uint64_t* rows_ready = sc_done + 1;   // [2]
  uint64_t* red_full = rows_ready + 2;  // [2] a [128][32] f32 dQ^T chunk is staged in buffer b
  uint64_t* red_free = red_full + 2;    // [2] buffer b's previous TMA reduce has finished reading it
  uint64_t* wo_full = red_free + 2;     // [2] the weight warps have staged dV (0), dK (1) (bf16 gradients)
  uint64_t* dv_done = wo_full + 2;      // the last dV product has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Head-dim half of dK, dV, dQ at D = 256 (two CTAs per key tile); key tile
  // 0 first (seen by the most rows).
  const int h = L::kSplit == 2 ? static_cast<int>(blockIdx.x & 1u) : 0;
  const int blk = L::kSplit == 2 ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  int kt, bkv;
  bwd_block_tile(p, blk, kt, bkv);
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
    for (int st = 0; st < STAGES; ++st) {
      mbar_init(&stage_full[st], 1);
      mbar_init(&stage_empty[st], 1);
      mbar_init(&q_full[st], 1);
      mbar_init(&q_empty[st], 1);
    }
    for (int b2 = 0; b2 < 2; ++b2) {
      mbar_init(&scores_full[b2], 1);
    }
    mbar_init(ds_full, 8);
    mbar_init(dq_full, 1);
    mbar_init(&dq_free[0], 4);
    mbar_init(&dq_free[1], 4);
    mbar_init(dkv_done, 1);
    mbar_init(sc_done, 1);
    mbar_init(&rows_ready[0], BQ);
    mbar_init(&rows_ready[1], BQ);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&red_full[i], 128);
      mbar_init(&red_free[i], 1);
    }
    mbar_init(&wo_full[0], 8);
    mbar_init(&wo_full[1], 8);
    mbar_init(dv_done, 1);
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
      int n_ld = 0;  // items loaded
      for (int n = 0; n < n_items; ++n) {
        const int bh = item_bh(n), q0 = item_q0(n);
        const int st = n % STAGES;
        uint8_t* stage = smem + L::kQOff + st * L::kStage;
        const uint32_t par = ((n / STAGES) & 1) ^ 1;
        if (!mbar_wait(&stage_empty[st], par, 70)) break;
        mbar_expect_tx(&stage_full[st], L::kSplitOps ? L::kQTile : 2 * L::kQTile);
        // dO first: the item's first product (dP^T) reads it.
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(stage + L::kQTile + c * (BQ * 128), &tmDO, &stage_full[st], c * 64, q0, bh);
        uint64_t* qbar = &stage_full[st];
        if (L::kSplitOps) {
          if (!mbar_wait(&q_empty[st], par, 71)) {
            n_ld = n;  // dO of item n is in flight: drained below with Q not issued
            mbar_wait(&stage_full[st], (n / STAGES) & 1, 74);
            break;
          }
          qbar = &q_full[st];
          mbar_expect_tx(qbar, L::kQTile);
        }
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(stage + c * (BQ * 128), &tmQ, qbar, c * 64, q0, bh);
        n_ld = n + 1;
      }
      // Drain: never leave the CTA with a copy still writing shared memory
      // (a load is issued only once the one STAGES earlier was consumed).
      mbar_wait(kv_full, 0, 72);
      for (int it = max(0, n_ld - STAGES); it < n_ld; ++it) {
        mbar_wait(&stage_full[it % STAGES], (it / STAGES) & 1, 73);
        if (L::kSplitOps) mbar_wait(&q_full[it % STAGES], (it / STAGES) & 1, 73);
      }
    }
    __syncwarp();
  } else if (warp == 1 || warp == 14) {
    // ---------------------------------------------------------------- MMA issuers
    // Warp 1 issues every item's score products (dP^T, S^T), warp 14 its
    // gradient products (dQ^T, dV, dK), each from one thread: a thread that
    // blocks on a full tensor pipe or on a barrier does not hold up the
    // other's instructions.  Products of different threads are not ordered,
    // so every reuse of a slot waits for the barrier of its last reader.
    if (lane == 0 && n_items > 0) {
      constexpr uint32_t kIdS = idesc_bf16_f32(128, BQ, 0, 0);   // S^T, dP^T: K-major A and B, N = 64
      constexpr uint32_t kIdG = idesc_bf16_f32(128, 128, 0, 1);  // dV_h, dK_h: A from TMEM, B MN-major
      constexpr uint32_t kIdQ = idesc_bf16_f32(128, BQ, 1, 1);   // dQ^T_h: A (K_h^T), B (dS^T) MN-major
      const uint64_t dK_a = sdesc_sw128(sbase + L::kKOff, 16, 1024);
      const uint64_t dV_a = sdesc_sw128(sbase + L::kVOff, 16, 1024);
      // Head-dim half h: boxes 2h, 2h + 1 of K (16 KB apart) and of Q, dO (8 KB apart).
      const uint64_t dKh_mn = sdesc_sw128(sbase + L::kKOff + h * 2 * (128 * 128), 128 * 128, 1024);
      const uint64_t dS_mn = sdesc_sw128(sbase + L::kDSOff, BQ * 128, 1024);
      bool ok = mbar_wait(kv_full, 0, 75);
      if (ok) tc_fence_after();
      if (warp == 1) {
        // Score products of item m into slot m & 1: dP^T = V dO^T, then
        // S^T = K Q^T (K = D).  The slot last held item m - 2: its S^T
        // columns took dQ^T_{m-2}, which must have been read out; its dP^T
        // columns held P^T and dS^T of m - 2, read by the dV and dK products
        // of m - 2 (waited for here with more than two stages; with one or
        // two, the load of item m waited for them already).
        for (int m = 0; ok && m < n_items; ++m) {
          const int st = m % STAGES;
          const uint32_t par = (m / STAGES) & 1;
          const int b2 = m & 1;
          if (m >= 2) {
            ok = mbar_wait(&dq_free[b2], ((m - 2) >> 1) & 1, 79);
            if (!ok) break;
            if (STAGES > 2) {
              ok = mbar_wait(&stage_empty[(m - 2) % STAGES], ((m - 2) / STAGES) & 1, 89);
              if (!ok) break;
            }
          }
          const uint32_t qs = sbase + L::kQOff + st * L::kStage;
          const uint64_t dQ_b = sdesc_sw128(qs, 16, 1024);
          const uint64_t dO_b = sdesc_sw128(qs + L::kQTile, 16, 1024);
          ok = mbar_wait(&stage_full[st], par, 76);  // dO (and Q unless split)
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t oa = static_cast<uint64_t>(((kk >> 2) * (128 * 128) + (kk & 3) * 32) >> 4);
            const uint64_t ob = static_cast<uint64_t>(((kk >> 2) * (BQ * 128) + (kk & 3) * 32) >> 4);
            umma_bf16_ss(tmem + L::kColDP + b2 * BQ, dV_a + oa, dO_b + ob, kIdS, kk > 0);
          }
          if (L::kSplitOps) {
            ok = mbar_wait(&q_full[st], par, 77);
            if (!ok) break;
            tc_fence_after();
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t oa = static_cast<uint64_t>(((kk >> 2) * (128 * 128) + (kk & 3) * 32) >> 4);
            const uint64_t ob = static_cast<uint64_t>(((kk >> 2) * (BQ * 128) + (kk & 3) * 32) >> 4);
            umma_bf16_ss(tmem + L::kColS + b2 * BQ, dK_a + oa, dQ_b + ob, kIdS, kk > 0);
          }
          umma_commit(&scores_full[b2]);
        }
        // Every product of this thread completes before the CTA frees the
        // tensor memory (also when a wait above gave up).
        umma_commit(sc_done);
        mbar_wait(sc_done, 0, 91);
      } else {
        for (int n = 0; ok && n < n_items; ++n) {
          const int st = n % STAGES;
          const int b2 = n & 1;
          const uint32_t qs = sbase + L::kQOff + st * L::kStage;
          const uint64_t dQh_mn = sdesc_sw128(qs + h * 2 * (BQ * 128), BQ * 128, 1024);
          const uint64_t dOh_mn = sdesc_sw128(qs + L::kQTile + h * 2 * (BQ * 128), BQ * 128, 1024);
          if (n >= 1) {
            // dQ^T_{n-1} has been read out before dQ^T_n is issued: once it
            // is, the read-out could see dq_full complete twice and the
            // phase parity would no longer tell the two apart.
            ok = mbar_wait(&dq_free[(n - 1) & 1], ((n - 1) >> 1) & 1, 90);
            if (!ok) break;
          }
          ok = mbar_wait(ds_full, n & 1, 78);
          if (!ok) break;
          tc_fence_after();
          // dQ^T_h = K_h^T dS^T (K = 128 keys) into the S^T columns of slot
          // n & 1 (the weights have read S^T_n), first, so that its read-out
          // overlaps the dV and dK products.
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t o = static_cast<uint64_t>((kk * (16 * 128)) >> 4);
            umma_bf16_ss(tmem + L::kColS + b2 * BQ, dKh_mn + o, dS_mn + o, kIdQ, kk > 0);
          }
          umma_commit(dq_full);
          // dV_h += P^T dO_h, dK_h += dS^T Q_h (K = 64 queries; the 16
          // queries of step kk lie in query half kk / 2: P^T at columns
          // 32 (kk / 2) + 16 + 8 (kk % 2) of the dP^T slot, dS^T at
          // 32 (kk / 2) + 8 (kk % 2)).
          const uint32_t dp_slot = tmem + L::kColDP + b2 * BQ;
#pragma unroll
          for (int kk = 0; kk < BQ / 16; ++kk) {
            const uint64_t o = static_cast<uint64_t>((kk * (16 * 128)) >> 4);
            const uint32_t pcol = (kk >> 1) * 32 + 16 + (kk & 1) * 8;
            umma_bf16_ts(tmem + L::kColDV, dp_slot + pcol, dOh_mn + o, kIdG, (n > 0 || kk > 0) ? 1u : 0u);
          }
          if (L::kSplitOps) umma_commit(&stage_empty[st]);  // dO's last reader
          if (n == n_items - 1) umma_commit(dv_done);        // dV is final: its write-out may start
#pragma unroll
          for (int kk = 0; kk < BQ / 16; ++kk) {
            const uint64_t o = static_cast<uint64_t>((kk * (16 * 128)) >> 4);
            const uint32_t dcol = (kk >> 1) * 32 + (kk & 1) * 8;
            umma_bf16_ts(tmem + L::kColDK, dp_slot + dcol, dQh_mn + o, kIdG, (n > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(L::kSplitOps ? &q_empty[st] : &stage_empty[st]);
        }
        umma_commit(dkv_done);
        mbar_wait(dkv_done, 0, 80);
      }
    }
    __syncwarp();
  } else if (warp >= 10 && warp < 14) {
    // ---------------------------------------------------------------- dQ^T read-out
    // dQ^T of item m (TMEM lane = head-dim row of half h, in the S^T columns
    // of slot m & 1), 32 query columns at a time: scaled and staged as
    // [32 queries][128 head-dim columns] f32 -- the accumulator's own [q][d]
    // layout (for a fixed query the warp's lanes write 32 consecutive
    // floats) -- and one thread adds the chunk into the f32 accumulator with a
    // TMA reduce.  A buffer is written again once its previous reduce has read
    // it (the issuing thread waits for that read only then, so reduces
    // overlap the next chunks).
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const bool issuer = warp == 10 && lane == 0;
    bool ok = true;
    for (int m = 0; ok && m < n_items; ++m) {
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(dq_full, m & 1, 85));
      if (!ok) break;
      tc_fence_after();
      uint32_t v[2][32];
      tmem_ld32x2(lane_base + L::kColS + (m & 1) * BQ, v[0], lane_base + L::kColS + (m & 1) * BQ + 32, v[1]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&dq_free[m & 1]);
      const int bh = item_bh(m), q0 = item_q0(m);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int b = L::kNumStg == 2 ? c : 0;
        const int use = L::kNumStg == 2 ? m : 2 * m + c;  // uses of buffer b so far
        if (use > 0) {
          if (issuer) {
            // The reduce that last used buffer b is the latest but one of this
            // thread's (two buffers) or its latest (one buffer).
            if (L::kNumStg == 2) bulk_wait_read<1>();
            else bulk_wait_read<0>();
            mbar_arrive(&red_free[b]);
          }
          ok = __all_sync(0xFFFFFFFFu, mbar_wait(&red_free[b], (use - 1) & 1, 86));
          if (!ok) break;
        }
        const uint32_t stg = sbase + L::kStgOff + b * 16384 + row * 4;
#pragma unroll
        for (int q = 0; q < 32; ++q) st_shared_f32(stg + q * 512, __uint_as_float(v[c][q]) * p.scale);
        fence_proxy_async_smem();
        mbar_arrive(&red_full[b]);
        if (issuer) {
          if (!mbar_wait(&red_full[b], use & 1, 87)) {
            ok = false;
          } else {
            tma_reduce_add_3d(&tmDQ, smem + L::kStgOff + b * 16384, h * 128, q0 + c * 32, bh);
            bulk_commit();
          }
        }
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (!ok) break;
      }
    }
    // Every dQ reduce of this CTA must have read its staging buffer before the
    // CTA (and its shared memory) ends; the global adds complete with the grid.
    if (issuer) bulk_wait_read<0>();
  } else {
    // ---------------------------------------------------------------- key rows: the weights
    const int quarter = warp & 3;             // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;         // query columns [32 half, 32 half + 32) of the item
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const int kj = k0 + row;                  // this thread's key
    const int c0 = half * 32;
    const bool row_writer = half == 0 && row < BQ;
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
      const int b2 = n & 1;
      const uint32_t slot_par = (n >> 1) & 1;
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
      int c_hi = p.Nq - q0;
      const int c_lo = p.causal ? kj - diag - q0 : -0x7FFFFFFF;
      if (p.window_left > 0) c_hi = min(c_hi, kj - diag + p.window_left - q0);  // left window
      const bool key_ok = kj < p.Nk;
      const bool masked = !(key_ok && c_lo <= c0 && c_hi >= c0 + 32);
      // The bias of this key row's 32 query columns, loaded before the wait
      // for the scores so that the loads are in flight meanwhile.
      float cb[BIAS ? 32 : 1];
      if constexpr (BIAS) {
        const BwdBiasRow br = bwd_bias_row(p, bh, q0, kj);
#pragma unroll
        for (int e = 0; e < 32; ++e) cb[e] = bwd_bias_at(br, c0 + e, key_ok, c_lo, c_hi);
        // The next item's dense-bias lines of this warp's 32 keys (one query
        // row per lane) into L2, so that its loads wait on L2 instead of DRAM.
        if (p.bias != nullptr && n + 1 < n_items) {
          const int qn = item_q0(n + 1) + c0 + lane;
          if (qn < p.Nq && kj - lane < p.Nk) {
            const BwdBiasRow bn = bwd_bias_row(p, item_bh(n + 1), item_q0(n + 1), kj - lane);
            prefetch_l2(bn.brow + static_cast<long long>(c0 + lane) * bn.bstride);
          }
        }
      }
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(&scores_full[b2], slot_par, 82));
      if (!ok) break;
      tc_fence_after();
      const uint32_t dp_cols = lane_base + L::kColDP + b2 * BQ + c0;
      uint32_t dp[32], sv[32];
      tmem_ld32x2(dp_cols, dp, lane_base + L::kColS + b2 * BQ + c0, sv);
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
            x0 += cb[e + u];
            x1 += cb[e + u + 1];
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
      // dS^T and P^T over this half's dP^T columns of the slot.
      tmem_st16(dp_cols, dw);
      tmem_st16(dp_cols + 16, pw);
      if (n > 0) {
        // dS^T into shared memory once the previous item's dQ^T product, its
        // other reader, has completed (row `row`, 16-byte units 4 half ..
        // 4 half + 3 in the 128-byte swizzle).
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(dq_full, (n - 1) & 1, 84));
        if (!ok) break;
      }
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
    }

    // dK_h, dV_h rows of this key (zeros when no query row sees the tile):
    // this thread's 64 of the CTA's 128 head-dim columns.  The tensor-memory
    // loads run on every lane; only the stores depend on the key being < Nk.
    if (ok && !p.g_f32 && n_items > 0) {
      // bf16 gradients, dV first (its last product completes before dK's):
      // each thread stages its key row's 64 columns of dV_h, then of dK_h, as
      // bf16 in the Q/dO ring ([128 keys][64 columns] boxes, 128-byte
      // swizzle, two per tensor), and one thread writes each tensor's boxes
      // with TMA stores as soon as they are staged (rows past Nk are not
      // written).  dV goes where the last item's dK product cannot be
      // reading: the next stage of the ring (two or more stages) or the dO
      // half of the one stage (dO's last reader, dV, is done); dK, staged
      // once every product has completed, takes the remaining 32 KB.
      const int last = n_items - 1;
      const uint32_t st_off[2] = {
          static_cast<uint32_t>(STAGES == 1 ? L::kQTile : ((last + 1) % STAGES) * L::kStage),
          static_cast<uint32_t>(STAGES == 1 ? 0 : ((last + 2) % STAGES) * L::kStage)};
#pragma unroll 1
      for (int which = 0; which < 2 && ok; ++which) {
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(which == 0 ? dv_done : dkv_done, 0, which == 0 ? 93 : 88));
        if (!ok) break;
        tc_fence_after();
        const uint32_t col = which == 0 ? L::kColDV : L::kColDK;
        const float mul = which == 0 ? 1.f : p.scale;
        const uint32_t box = sbase + L::kQOff + st_off[which] + half * (128 * 128) + row * 128;
        uint32_t v[2][32];
        tmem_ld32x2(lane_base + col + half * 64, v[0], lane_base + col + half * 64 + 32, v[1]);
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int x = 8 * u;
            st_shared_v4(box + (((c2 * 4 + u) ^ (row & 7)) << 4),
                         pack_bf16(__uint_as_float(v[c2][x]) * mul, __uint_as_float(v[c2][x + 1]) * mul),
                         pack_bf16(__uint_as_float(v[c2][x + 2]) * mul, __uint_as_float(v[c2][x + 3]) * mul),
                         pack_bf16(__uint_as_float(v[c2][x + 4]) * mul, __uint_as_float(v[c2][x + 5]) * mul),
                         pack_bf16(__uint_as_float(v[c2][x + 6]) * mul, __uint_as_float(v[c2][x + 7]) * mul));
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&wo_full[which]);
        if (threadIdx.x == 64 && mbar_wait(&wo_full[which], 0, 92)) {
#pragma unroll
          for (int bx = 0; bx < 2; ++bx)
            tma_store_3d(which == 0 ? &tmDVo : &tmDKo, smem + L::kQOff + st_off[which] + bx * (128 * 128),
                         h * 128 + bx * 64, k0, bkv);
          bulk_commit();
        }
      }
      // The boxes are read before the CTA ends; the writes complete with the grid.
      if (threadIdx.x == 64) bulk_wait_read<0>();
    } else if (ok) {
      // f32 gradients (or a key tile no query row sees: zeros), stored
      // directly from registers once every product has completed.
      if (n_items > 0) {
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(dkv_done, 0, 88));
        if (ok) tc_fence_after();
      }
    }
    if (ok && (p.g_f32 || n_items == 0)) {
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

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace attn
