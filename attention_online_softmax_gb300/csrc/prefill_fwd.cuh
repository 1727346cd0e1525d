// Fused attention forward (prefill) for sm_103a.
//
// A CTA computes NQ 128-row query tiles (NQ = 2 for d <= 128, 1 for d = 256)
// of one (batch, query head) against the key/value tiles those rows may see,
// following the block recurrence of "Compilers and Kernels", section
// "FlashAttention changes the algorithm around IO": for each key block B_t the
// row state (m, l, o) is updated by
//     m_t = max(m_{t-1}, b_t),  alpha_t = exp(m_{t-1} - m_t),
//     l_t = alpha_t l_{t-1} + sum exp(S - m_t),  o_t = alpha_t o_{t-1} + sum exp(S - m_t) v,
// and O = o_T / l_T, LSE = m_T + ln l_T at the end.  Scores never leave the SM.
//
// Roles (64 + 128*NQ threads):
//   warp 0        TMA producer: the NQ query tiles once, then K_t, V_t tiles
//                 (shared by all query tiles of the CTA) into a STAGES-deep
//                 shared-memory ring (128-byte swizzle), gated by mbarriers.
//   warp 1        allocates tensor memory; one thread issues tcgen05.mma:
//                 S_j = Q_j K_t^T (smem x smem) into TMEM, then
//                 O_j += P_j V_t with P_j read from TMEM (tmem x smem).
//   warps 2..     one softmax warpgroup per query tile, one thread per row:
//                 reads S from TMEM, applies the mask, updates the running max,
//                 writes P = 2^(x - m) as bf16 back over S in TMEM, rescales O
//                 in TMEM when the max moved, and writes O / l and LSE.
//
// Tensor memory (512 columns): O_j at columns [j*D, (j+1)*D); two S slots of
// 128 columns after them.  With NQ = 2 slot j belongs to query tile j and the
// MMA order PV_A(t-1), S_A(t), PV_B(t-1), S_B(t) lets one warpgroup's softmax
// overlap the other tile's MMAs.  With NQ = 1 the slots alternate over key
// tiles: S(t+1) is computed while tile t is softmaxed.  P (bf16, 64 columns)
// overwrites the first half of its S slot; tcgen05 MMAs from one thread run in
// issue order, so the next S into that slot is issued after the P V product.
//
// Work is in base 2: x = s * scale * log2(e), p = 2^(x - m); the running
// reference max only moves when a tile's max exceeds it by more than
// kRescaleLog2 (2^8) -- exact for any reference (numerator and denominator
// share it) while bounding p <= 256, so most tiles skip the O rescale.  O is
// normalised by the sum of the bf16-rounded p (the weights the P V product
// used); LSE uses the sum of the unrounded p.  The scale must be positive (the
// host checks it), so the max of the raw scores gives the max of the scaled.
#pragma once

#include "ptx.cuh"

#ifndef ATTN_MMA_WAIT
#define ATTN_MMA_WAIT mbar_wait
#endif
#ifndef ATTN_SOFTMAX_WAIT
#define ATTN_SOFTMAX_WAIT mbar_wait
#endif

namespace attn {

constexpr int kBM = 128;  // query rows per tile (TMEM lanes)
constexpr int kBN = 128;  // keys per tile
constexpr float kRescaleLog2 = 8.0f;

struct PrefillParams {
  void* o;
  float* lse;
  int B, Hq, Hkv, Nq, Nk;
  int causal;
  int o_f32;
  int n_units;       // CTAs per (batch, head): ceil(Nq / (128 * NQ))
  int group;         // (batch, head) pairs scheduled together, longest units first
  float scale_log2;  // scale * log2(e), > 0
};

template <int D, int NQ, int STAGES>
struct PrefillLayout {
  static constexpr int kThreads = 64 + 128 * NQ;
  static constexpr int kQBytes = kBM * D * 2;
  // K and V tiles stream in items of up to 128 head-dim columns (kH items per
  // tile), so with d = 256 a 64 KB tile occupies two 32 KB ring stages and
  // loading the next tile overlaps the current one's MMAs.
  static constexpr int kDI = D < 128 ? D : 128;  // head-dim columns per item
  static constexpr int kH = D / kDI;             // items per K (or V) tile
  static constexpr int kKVBytes = kBN * kDI * 2; // one ring stage
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = kQOff + NQ * kQBytes;
  static constexpr int kBarOff = kKVOff + STAGES * kKVBytes;
  // q_full, kv_full[S], kv_empty[S], s_full[2], p_full[2], pv_done, o_done[2], mma_drain
  static constexpr int kNumBars = 1 + 2 * STAGES + 2 + 2 + 1 + 2 + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kMiscOff + 16;
  static constexpr int kAlloc = kBytes + 1024;  // room to align the dynamic base to 1024
  static constexpr int kTmemCols = 512;
  static constexpr int kSCol = NQ * D;          // first S slot column
  static_assert(NQ * D + 2 * kBN <= kTmemCols, "tensor memory budget");
  static_assert(kAlloc <= 232448, "shared memory budget");
  static_assert(D % 64 == 0, "head dim");
  static_assert(NQ == 1 || NQ == 2, "query tiles per CTA");
};

template <int D, int NQ, int STAGES>
__global__ void __launch_bounds__(PrefillLayout<D, NQ, STAGES>::kThreads, 1)
    prefill_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
  using L = PrefillLayout<D, NQ, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const uint32_t sbase = smem_u32(smem);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = kv_full + STAGES;
  uint64_t* s_full = kv_empty + STAGES;
  uint64_t* p_full = s_full + 2;
  uint64_t* pv_done = p_full + 2;
  uint64_t* o_done = pv_done + 1;
  uint64_t* mma_drain = o_done + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Flat grid in groups of `group` (batch, head) pairs; inside a group the
  // blocks run longest causal unit first across all its heads (the block
  // scheduler then packs the uneven causal units well), while the group's
  // K/V stay small enough to be reused from L2.
  const int BH = p.B * p.Hq;
  const int per_group = p.group * p.n_units;
  const int grp = static_cast<int>(blockIdx.x) / per_group;
  const int idx = static_cast<int>(blockIdx.x) - grp * per_group;
  const int gsize = min(p.group, BH - grp * p.group);
  const int rank = gsize > 0 ? idx / gsize : p.n_units;
  const int bh = grp * p.group + (idx - rank * gsize);
  const int unit = p.n_units - 1 - rank;
  if (gsize <= 0 || bh >= BH || unit < 0) return;  // never taken with the host's grid
  const int b = bh / p.Hq;
  const int h = bh - b * p.Hq;
  const int kvh = b * p.Hkv + h / (p.Hq / p.Hkv);
  const int q0 = unit * (kBM * NQ);
  const int diag = p.Nk - p.Nq;  // key j allowed for row i iff j <= i + diag (causal)

  // Key tiles each query tile needs (0 for a tile past Nq or fully masked).
  int ntile[NQ];
  int T = 0;
#pragma unroll
  for (int j = 0; j < NQ; ++j) {
    const int r0 = q0 + j * kBM;
    int kend = 0;
    if (r0 < p.Nq) {
      kend = p.Nk;
      if (p.causal) kend = min(p.Nk, min(r0 + kBM, p.Nq) - 1 + diag + 1);
    }
    ntile[j] = kend > 0 ? (kend + kBN - 1) / kBN : 0;
    T = max(T, ntile[j]);
  }

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 4);
      mbar_init(&o_done[i], 1);
    }
    mbar_init(pv_done, 1);
    mbar_init(mma_drain, 1);
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
    if (lane == 0 && T > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_expect_tx(q_full, NQ * L::kQBytes);
#pragma unroll
      for (int j = 0; j < NQ; ++j)
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + L::kQOff + j * L::kQBytes + c * (kBM * 128), &tmQ, q_full, c * 64, q0 + j * kBM,
                      bh);
      int issued = 0;
      for (int item = 0; item < 2 * L::kH * T; ++item) {
        const int st = item % STAGES;
        if (!mbar_wait(&kv_empty[st], ((item / STAGES) & 1) ^ 1, 1)) break;
        mbar_expect_tx(&kv_full[st], L::kKVBytes);
        const int t = item / (2 * L::kH);
        const int kind = (item / L::kH) & 1;  // 0: K, 1: V
        const int hh = item % L::kH;          // which 128-column part of the head dim
        const CUtensorMap* map = kind ? &tmV : &tmK;
#pragma unroll
        for (int c = 0; c < L::kDI / 64; ++c)
          tma_load_3d(smem + L::kKVOff + st * L::kKVBytes + c * (kBN * 128), map, &kv_full[st],
                      hh * L::kDI + c * 64, t * kBN, kvh);
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
    if (lane == 0 && T > 0) {
      constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, kBN, 0, 0);      // Q K-major, K K-major
      constexpr uint32_t kIdescO = idesc_bf16_f32(kBM, L::kDI, 0, 1);   // P K-major (TMEM), V MN-major
      bool ok = mbar_wait(q_full, 0, 10);

      // Descriptor bases, computed once: within a group only compile-time
      // offsets are added (the 14-bit address field cannot carry: every
      // shared-memory address is below 256 KB), so the issuing thread spends
      // its time issuing MMAs rather than building descriptors.
      const uint64_t dq0 = sdesc_sw128(sbase + L::kQOff, 16, 1024);
      const uint64_t dkv0 = sdesc_sw128(sbase + L::kKVOff, 16, 1024);
      const uint64_t dv0 = sdesc_sw128(sbase + L::kKVOff, kBN * 128, 1024);
      auto item_of = [](int t, int kind, int hh) { return t * 2 * L::kH + kind * L::kH + hh; };
      auto wait_item = [&](int item, int where) {
        return ATTN_MMA_WAIT(&kv_full[item % STAGES], (item / STAGES) & 1, where);
      };
      // S_j(t) = Q_j K_t^T into S slot `slot`; waits for each K item in turn.
      auto issue_s = [&](int j, int slot, int t, bool wait) -> bool {
        const uint64_t da = dq0 + static_cast<uint64_t>((j * L::kQBytes) >> 4);
        const uint32_t dst = tmem + L::kSCol + slot * kBN;
#pragma unroll
        for (int hh = 0; hh < L::kH; ++hh) {
          const int item = item_of(t, 0, hh);
          if (wait) {
            if (!wait_item(item, 13)) return false;
            tc_fence_after();
          }
          const uint64_t db = dkv0 + static_cast<uint64_t>(((item % STAGES) * L::kKVBytes) >> 4);
#pragma unroll
          for (int k2 = 0; k2 < L::kDI / 16; ++k2) {
            const int kk = hh * (L::kDI / 16) + k2;
            const uint64_t oa = static_cast<uint64_t>(((kk >> 2) * (kBM * 128) + (kk & 3) * 32) >> 4);
            const uint64_t ob = static_cast<uint64_t>(((k2 >> 2) * (kBN * 128) + (k2 & 3) * 32) >> 4);
            umma_bf16_ss(dst, da + oa, db + ob, kIdescS, kk > 0);
          }
        }
        return true;
      };
      // O_j (+)= P_j V_t: one N = kDI product per V item.
      auto issue_pv = [&](int j, int slot, int t, bool wait) -> bool {
        const uint32_t pa = tmem + L::kSCol + slot * kBN;
#pragma unroll
        for (int hh = 0; hh < L::kH; ++hh) {
          const int item = item_of(t, 1, hh);
          if (wait) {
            if (!wait_item(item, 11)) return false;
            tc_fence_after();
          }
          const uint64_t db = dv0 + static_cast<uint64_t>(((item % STAGES) * L::kKVBytes) >> 4);
          const uint32_t dst = tmem + j * D + hh * L::kDI;
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            umma_bf16_ts(dst, pa + kk * 8, db + static_cast<uint64_t>((kk * (16 * 128)) >> 4), kIdescO,
                         (t > 0 || kk > 0) ? 1u : 0u);
        }
        return true;
      };
      auto release = [&](int t, int kind) {
#pragma unroll
        for (int hh = 0; hh < L::kH; ++hh) umma_commit(&kv_empty[item_of(t, kind, hh) % STAGES]);
      };

      for (int t = 0; ok && t <= T; ++t) {
        if (NQ == 2) {
          // PV_A(t-1), S_A(t), PV_B(t-1), S_B(t); K/V items are waited for by
          // their first user and released after their last.
          bool waitedV = false, waitedK = false;
#pragma unroll
          for (int j = 0; j < NQ; ++j) {
            if (t >= 1 && t - 1 < ntile[j]) {
              ok = ATTN_MMA_WAIT(&p_full[j], (t - 1) & 1, 12);
              if (!ok) break;
              tc_fence_after();
              ok = issue_pv(j, j, t - 1, !waitedV);
              if (!ok) break;
              waitedV = true;
              if (t - 1 == ntile[j] - 1) umma_commit(&o_done[j]);
            }
            if (t < ntile[j]) {
              ok = issue_s(j, j, t, !waitedK);
              if (!ok) break;
              waitedK = true;
              umma_commit(&s_full[j]);
            }
          }
          if (!ok) break;
          if (waitedV) release(t - 1, 1);
          if (waitedK) release(t, 0);
        } else {
          // S(t) into slot t&1 (overlaps the softmax of tile t-1), then PV(t-1).
          if (t < T) {
            ok = issue_s(0, t & 1, t, true);
            if (!ok) break;
            umma_commit(&s_full[t & 1]);
            release(t, 0);
          }
          if (t >= 1) {
            ok = ATTN_MMA_WAIT(&p_full[(t - 1) & 1], ((t - 1) >> 1) & 1, 12);
            if (!ok) break;
            tc_fence_after();
            ok = issue_pv(0, (t - 1) & 1, t - 1, true);
            if (!ok) break;
            umma_commit(pv_done);
            release(t - 1, 1);
            if (t - 1 == T - 1) umma_commit(&o_done[0]);
          }
        }
      }
      if (!ok) report_error(6 /* ATTN_ERR_TIMEOUT */, 16, 0);
      // Every MMA this thread issued must be complete before TMEM is freed.
      umma_commit(mma_drain);
      mbar_wait(mma_drain, 0, 15);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- softmax warpgroups
    const int j = (warp - 2) >> 2;           // query tile of this warpgroup
    const int quarter = warp & 3;            // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;     // row within the tile
    const int r0 = q0 + j * kBM;
    const int qrow = r0 + row;
    const int nt = ntile[j];
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t o_cols = lane_base + j * D;
    const float sl = p.scale_log2;
    // l sums the exact weights (for LSE); lr sums the bf16-rounded weights the
    // P V product uses, so O = o / lr is an exact convex combination of V rows
    // before output rounding.
    float m_ref = -INFINITY;
    float l0 = 0.f, l1 = 0.f, lr0 = 0.f, lr1 = 0.f;
    bool ok = true;

    for (int t = 0; t < nt; ++t) {
      const int slot = NQ == 2 ? j : (t & 1);
      const uint32_t s_par = NQ == 2 ? (t & 1) : ((t >> 1) & 1);
      ok = __all_sync(0xFFFFFFFFu, ATTN_SOFTMAX_WAIT(&s_full[slot], s_par, 20));
      if (!ok) break;
      tc_fence_after();
      uint32_t r[kBN];
      tmem_ld128(lane_base + L::kSCol + slot * kBN, r);

      // Row max of the raw scores (masked keys -> -inf); scale > 0 keeps the
      // order, so the scaled max is mx * sl.
      const int k0 = t * kBN;
      const bool need_mask = (k0 + kBN > p.Nk) || (p.causal && (k0 + kBN - 1 > r0 + diag));
      if (need_mask) {
        const int lim = (p.causal ? min(p.Nk - 1, qrow + diag) : p.Nk - 1) - k0;
#pragma unroll
        for (int c = 0; c < kBN; ++c)
          if (c > lim) r[c] = 0xFF800000u;  // -inf
      }
      float mx[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) mx[i] = -INFINITY;
#pragma unroll
      for (int c = 0; c < kBN; c += 8) {
        const int a = (c >> 3) & 3;
        mx[a] = fmax3(mx[a], __uint_as_float(r[c]), __uint_as_float(r[c + 1]));
        mx[a] = fmax3(mx[a], __uint_as_float(r[c + 2]), __uint_as_float(r[c + 3]));
        mx[a] = fmax3(mx[a], __uint_as_float(r[c + 4]), __uint_as_float(r[c + 5]));
        mx[a] = fmax3(mx[a], __uint_as_float(r[c + 6]), __uint_as_float(r[c + 7]));
      }
      const float mt = fmaxf(fmax3(mx[0], mx[1], mx[2]), mx[3]) * sl;
      const float m_new = fmaxf(m_ref, mt);
      const bool rescale = m_new > m_ref + kRescaleLog2;
      float alpha = 1.f;
      if (rescale) {
        alpha = ex2(m_ref - m_new);  // 0 when m_ref = -inf
        m_ref = m_new;
        l0 *= alpha;
        l1 *= alpha;
        lr0 *= alpha;
        lr1 *= alpha;
      }
      const float neg_m = (m_ref == -INFINITY) ? 0.f : -m_ref;

      // p = 2^(s * sl - m): P as bf16 pairs, exact and rounded row sums.
      uint32_t pk[kBN / 2];
#pragma unroll
      for (int c = 0; c < kBN; c += 2) {
        float a0, a1;
        ffma2(a0, a1, __uint_as_float(r[c]), __uint_as_float(r[c + 1]), sl, sl, neg_m, neg_m);
        const float p0 = ex2(a0);
        const float p1 = ex2(a1);
        fadd2(l0, l1, l0, l1, p0, p1);
        const uint32_t w = pack_bf16(p0, p1);
        add_bf16x2(lr0, lr1, w);
        pk[c >> 1] = w;
      }

      if (t > 0 && __any_sync(0xFFFFFFFFu, rescale)) {
        if (NQ == 1) {
          // O holds tile t-1's contribution only once PV(t-1) is complete.
          ok = __all_sync(0xFFFFFFFFu, mbar_wait(pv_done, (t - 1) & 1, 21));
          if (!ok) break;
          tc_fence_after();
        }
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(o_cols + c * 32, o);
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float y0, y1;
            ffma2(y0, y1, __uint_as_float(o[i]), __uint_as_float(o[i + 1]), alpha, alpha, 0.f, 0.f);
            o[i] = __float_as_uint(y0);
            o[i + 1] = __float_as_uint(y1);
          }
          tmem_st32(o_cols + c * 32, o);
        }
      }
      // P over the first half of the S slot, then hand it to the MMA thread.
      tmem_st64(lane_base + L::kSCol + slot * kBN, pk);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[slot]);
    }

    if (ok && nt > 0) {
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(&o_done[j], 0, 22));
      if (ok) tc_fence_after();
    }
    // Every lane runs the (warp-collective) TMEM loads; only rows < Nq store.
    const bool store = qrow < p.Nq;
    if (ok) {
      const float lr = lr0 + lr1;
      const float l = l0 + l1;
      const float inv = (lr > 0.f) ? 1.f / lr : 0.f;
      const size_t row_off = (static_cast<size_t>(bh) * p.Nq + qrow) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        if (nt > 0) {
          tmem_ld32(o_cols + c * 32, o);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0u;
        }
        if (!store) continue;
        if (p.o_f32) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + row_off + c * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(__uint_as_float(o[4 * i]) * inv, __uint_as_float(o[4 * i + 1]) * inv,
                                 __uint_as_float(o[4 * i + 2]) * inv, __uint_as_float(o[4 * i + 3]) * inv);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + row_off + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int e = 8 * i;
            dst[i] = make_uint4(pack_bf16(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv),
                                pack_bf16(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv),
                                pack_bf16(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv),
                                pack_bf16(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv));
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
