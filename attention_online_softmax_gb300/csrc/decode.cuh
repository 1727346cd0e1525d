// Paged split-KV decode for sm_103a: one query row per (sequence, query head)
// against a paged KV cache, as a bandwidth-bound GEMV-class stage.
//
// Work item = (sequence, chunk of up to 256 cached tokens, group of hg
// key/value heads), ordered by chunk index from the last to the first: the
// slots past a sequence's end and the sequences' partial last chunks come
// first, and the launch ends on the uniform layer of first chunks, after which
// every sequence's merge runs at once.  Either one CTA per item slot (slots
// past a sequence's end exit at once), or a persistent grid (one or two CTAs
// per SM) in which CTA b starts on item b and takes the rest from a shared
// counter (sched_fetch), skipping chunks past a sequence's end.  One
// producer thread streams each item's cached tokens with TMA in boxes of
// [16 slots][hg heads][d] (first the K boxes, then the V boxes) into a ring
// of shared-memory stages that runs on across the items of a CTA; for page
// sizes above 16 a box is the 16-slot window of a page at the token's slot
// offset.  Compute warp w serves
// key/value head w / WPH of the group and GW of the query heads that share it
// (grouped-query attention: one read of K/V serves the whole group; a group
// of 16 query heads is split over two warps).  Lanes own 16-byte slices of a
// key row; partial dot products are reduced across the lanes of a row by a
// reduce-scatter over shuffles.  The chunk's scores stay in shared memory, so
// the chunk is softmaxed once (max, 2^(x - m), sum) and then the V boxes are
// accumulated.
//
// A sequence that fits one chunk is finished directly.  Otherwise each chunk
// stores its partial state as (O_c, lse_c) = (o / l, m + ln l) ("online
// softmax as a monoid", Tang abstract), and the warp that delivers the last
// chunk of a (sequence, head group, warp) merges them:
// LSE = logsumexp_c(lse_c), O = sum_c exp(lse_c - LSE) O_c -- the merge of
// partial states of the block recurrence in "Compilers and Kernels", section
// "FlashAttention changes the algorithm around IO", applied to whole chunks.
// Arrivals are counted in the workspace by epoch-tagged words (merge_arrive),
// so the merge needs no second kernel and no zeroed workspace.
#pragma once

#include "ptx.cuh"

namespace attn {

constexpr int kBox = 16;         // cached tokens per TMA box (one ring stage)
constexpr int kChunkMax = 256;   // tokens per work item, upper bound
constexpr int kMaxStages = 8;
constexpr int kItemQ = 4;        // depth of the in-CTA queue of work items
constexpr int kCntBits = 24;     // merge counter: arrivals in the low bits, the call's epoch above

struct DecodeParams {
  const uint16_t* q;
  const int32_t* block_table;
  const int32_t* seqlens;
  void* o;
  float* lse;
  float* ws_o;                  // [num_seqs][n_splits][Hq][D] chunk outputs O_c
  float* ws_lse;                // [num_seqs][n_splits][Hq]    chunk lse_c
  unsigned long long* ws_cnt;   // [num_seqs][ngroups][warps] merge counters (epoch << 24 | arrivals)
  unsigned long long* sched;    // this launch's work counter slot (sched_fetch); null: one item per CTA
  unsigned sched_tag;
  unsigned long long epoch;     // this call's merge epoch: nonzero, < 2^40
  int num_seqs, Hq, Hkv, num_pages, max_pages, max_seqlen, page_size;
  int chunk;      // tokens per work item: multiple of 16, <= kChunkMax
  int n_splits;   // ceil(max_seqlen / chunk), >= 1
  int hg;         // key/value heads per work item
  int ngroups;    // Hkv / hg
  int stages;     // shared-memory ring depth
  int stage_bytes;
  int o_f32;
  float scale_log2;
};

// Context length of `seq`, clamped to what the block table and max_seqlen
// allow (a length outside [0, cap] is reported when `report`).
__device__ __forceinline__ int decode_len(const DecodeParams& p, int seq, bool report) {
  int L = __ldg(p.seqlens + seq);
  const long long cap_ll = min(static_cast<long long>(p.max_seqlen), static_cast<long long>(p.max_pages) * p.page_size);
  const int cap = static_cast<int>(cap_ll);
  if (L < 0 || L > cap) {
    if (report) report_error(7 /* ATTN_ERR_BOUNDS */, seq, L);
    L = L < 0 ? 0 : cap;
  }
  return L;
}

template <int D, int GW>
struct DecodeShape {
  static constexpr int LPT = D / 8;            // lanes per key row (16 bytes each)
  static constexpr int TPP = 32 / LPT;         // key rows per pass of the warp
  static constexpr int PASSES = kBox / TPP;    // passes per box
  static constexpr int R0 = (2 * LPT) / GW;
  static constexpr int R = PASSES < (R0 > 0 ? R0 : 1) ? PASSES : (R0 > 0 ? R0 : 1);  // passes per reduction
  static constexpr int NV = R * GW;            // partial sums per lane per reduction
  static constexpr int LEVELS = LPT == 32 ? 5 : LPT == 16 ? 4 : 3;
  static constexpr int LOG_NV = NV >= 64 ? 6 : NV >= 32 ? 5 : NV >= 16 ? 4 : NV >= 8 ? 3 : NV >= 4 ? 2 : NV >= 2 ? 1 : 0;
  static constexpr int SCAT = LEVELS < LOG_NV ? LEVELS : LOG_NV;  // reduce-scatter levels
  static constexpr int KEEP = NV >> SCAT;      // sums a lane keeps
  static_assert(PASSES % R == 0, "reduction rounds");
  static_assert(D == 64 || D == 128 || D == 256, "head dim");
};

// Sum v[] across the LPT lanes that share a key row (lane bits below LPT).
// First reduce-scatter (each level halves the values a lane keeps), then plain
// butterflies once one value is left.  Afterwards lane `sub` holds the sums
// with indices [(sub >> (LEVELS - SCAT)) * KEEP, +KEEP).
template <int NV, int LPT, int SCAT, int LEVELS>
__device__ __forceinline__ void lane_reduce(float (&v)[NV], int lane) {
#pragma unroll
  for (int lev = 0; lev < SCAT; ++lev) {
    const int off = LPT >> (lev + 1);
    const int n = NV >> (lev + 1);
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < n; ++i) {
      const float send = upper ? v[i] : v[i + n];
      const float keep = upper ? v[i + n] : v[i];
      v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, off);
    }
  }
#pragma unroll
  for (int lev = SCAT; lev < LEVELS; ++lev) {
    const int off = LPT >> (lev + 1);
    v[0] += __shfl_xor_sync(0xFFFFFFFFu, v[0], off);
  }
}

// One arrival of a chunk at the merge counter of its (sequence, head group,
// warp); true for the arrival that completes `total`.  The word holds
// (epoch << 24) | arrivals of the call with that epoch; a word with another
// epoch (a former call's, or whatever the workspace held) counts as zero
// arrivals.  The last arrival resets the word to 0, so a replay of the same
// call (same epoch) starts from zero as well.  The compare-and-swap retries
// only when another arrival got in first (bounded all the same).
__device__ __forceinline__ bool merge_arrive(unsigned long long* cnt, unsigned long long epoch, int total) {
  unsigned long long old = atomicAdd(cnt, 0ull);
  for (int tries = 0; tries < (1 << 20); ++tries) {
    const unsigned long long arrived = (old >> kCntBits) == epoch ? (old & ((1ull << kCntBits) - 1)) : 0ull;
    const unsigned long long prev = atomicCAS(cnt, old, (epoch << kCntBits) | (arrived + 1));
    if (prev == old) {
      if (arrived + 1 != static_cast<unsigned long long>(total)) return false;
      atomicExch(cnt, 0ull);
      return true;
    }
    old = prev;
  }
  report_error(6 /* ATTN_ERR_TIMEOUT */, 61, total);
  return false;
}

// Merge the chunk partials of query heads [head0, head0 + GW) of `seq`: one
// warp, lanes own D/32 elements of every row.  The rows of U chunks of all GW
// heads are loaded together, so the walk over the chunks takes few L2 round
// trips.  Partials are read through L2 (ld.global.cg): other CTAs wrote them
// during this kernel.
template <int D, int GW>
__device__ __forceinline__ void merge_heads(const DecodeParams& p, int seq, int head0, int ns, int lane) {
  constexpr int E = D / 32;
  constexpr int U0 = 32 / (GW * E);
  constexpr int U = U0 < 1 ? 1 : (U0 > 4 ? 4 : U0);  // chunks whose rows are loaded together
  const size_t row0 = static_cast<size_t>(seq) * p.n_splits * p.Hq + head0;  // (chunk 0, head0)
  float m[GW];
#pragma unroll
  for (int g = 0; g < GW; ++g) m[g] = -INFINITY;
  for (int c = lane; c < ns; c += 32)
#pragma unroll
    for (int g = 0; g < GW; ++g) m[g] = fmaxf(m[g], __ldcg(p.ws_lse + row0 + static_cast<size_t>(c) * p.Hq + g));
#pragma unroll
  for (int g = 0; g < GW; ++g)
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m[g] = fmaxf(m[g], __shfl_xor_sync(0xFFFFFFFFu, m[g], off));
  // m = -inf only if every chunk was empty, which a multi-chunk sequence never is.
  float acc[GW][E], wsum[GW];
#pragma unroll
  for (int g = 0; g < GW; ++g) {
    wsum[g] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[g][e] = 0.f;
  }
  for (int c0 = 0; c0 < ns; c0 += 32) {
    const int cl = c0 + lane;
    float wl[GW];
#pragma unroll
    for (int g = 0; g < GW; ++g) {
      wl[g] = cl < ns ? ex2((__ldcg(p.ws_lse + row0 + static_cast<size_t>(cl) * p.Hq + g) - m[g]) *
                            1.4426950408889634f)
                      : 0.f;
      wsum[g] += wl[g];
    }
    const int nb = min(32, ns - c0);
    for (int k = 0; k < nb; k += U) {
      float v[U][GW][E];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = min(c0 + k + u, ns - 1);  // in range; weight 0 past the end
#pragma unroll
        for (int g = 0; g < GW; ++g) {
          const float* src = p.ws_o + (row0 + static_cast<size_t>(c) * p.Hq + g) * D + lane * E;
#pragma unroll
          for (int e = 0; e < E; e += 2) {
            const float2 x = __ldcg(reinterpret_cast<const float2*>(src + e));
            v[u][g][e] = x.x;
            v[u][g][e + 1] = x.y;
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int g = 0; g < GW; ++g) {
          float w = __shfl_sync(0xFFFFFFFFu, wl[g], (k + u) & 31);
          if (k + u >= nb) w = 0.f;
#pragma unroll
          for (int e = 0; e < E; ++e) acc[g][e] = fmaf(w, v[u][g][e], acc[g][e]);
        }
    }
  }
#pragma unroll
  for (int g = 0; g < GW; ++g) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) wsum[g] += __shfl_xor_sync(0xFFFFFFFFu, wsum[g], off);
    const float inv = 1.f / wsum[g];
    const size_t off = (static_cast<size_t>(seq) * p.Hq + head0 + g) * D + lane * E;
    if (p.o_f32) {
      float* dst = static_cast<float*>(p.o) + off;
#pragma unroll
      for (int e = 0; e < E; e += 2)
        *reinterpret_cast<float2*>(dst + e) = make_float2(acc[g][e] * inv, acc[g][e + 1] * inv);
    } else {
      uint32_t* dst = reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(p.o) + off);
#pragma unroll
      for (int e = 0; e < E; e += 2) dst[e / 2] = pack_bf16(acc[g][e] * inv, acc[g][e + 1] * inv);
    }
    if (lane == 0) p.lse[static_cast<size_t>(seq) * p.Hq + head0 + g] = m[g] + logf(wsum[g]);
  }
}

struct DecodeItem {
  int seq, chunk, group, len;  // seq -1: no work left (-2: the producer stopped after a timeout)
};

// Dynamic shared memory besides the ring: the scores, the barriers and the
// item queue, plus the slack for aligning the base to 1024 bytes.
__host__ __device__ constexpr int decode_fixed_bytes(int warps, int chunk, int gw) {
  return warps * chunk * gw * 4 + (2 * kMaxStages + 2 * kItemQ) * 8 + kItemQ * 16 + 1024;
}

// Up to four query heads per warp and d <= 128: two CTAs per SM (registers capped for it).
template <int D, int GW, int WPH>
__global__ void __launch_bounds__(288, (GW <= 4 && D <= 128) ? 2 : 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const DecodeParams p) {
  using S = DecodeShape<D, GW>;
  constexpr int G = GW * WPH;  // query heads per key/value head
  const int nw = p.hg * WPH;   // compute warps
  const int U = p.num_seqs * p.n_splits * p.ngroups;
  const int per_layer = p.num_seqs * p.ngroups;  // items of one chunk index

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const uint32_t sbase = smem_u32(smem);
  float* scores = reinterpret_cast<float*>(smem + p.stages * p.stage_bytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.stages * p.stage_bytes + nw * p.chunk * GW * 4);
  uint64_t* empty = full + kMaxStages;
  uint64_t* item_full = empty + kMaxStages;
  uint64_t* item_empty = item_full + kItemQ;
  DecodeItem* items = reinterpret_cast<DecodeItem*>(item_empty + kItemQ);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], nw);
    }
    for (int i = 0; i < kItemQ; ++i) {
      mbar_init(&item_full[i], 1);
      mbar_init(&item_empty[i], nw);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == nw) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const int ps = p.page_size;
      bool owned = false;
      bool ok = true;
      int box = 0;  // boxes issued (ring position, runs on across items)
      int n = 0;    // items published
      int w = static_cast<int>(blockIdx.x);  // first item: static (the grid is never larger than U)
      while (ok && w < U) {
        const int layer = w / per_layer;
        const int rem = w - layer * per_layer;
        const int ch = p.n_splits - 1 - layer;
        const int seq = rem / p.ngroups;
        const int grp = rem - seq * p.ngroups;
        const int L = decode_len(p, seq, ch == 0 && grp == 0);
        // Chunk 0 is always an item (a sequence of length 0 still gets O = 0,
        // LSE = -inf); later chunks only while they hold tokens.
        if (ch == 0 || ch * p.chunk < L) {
          const int slot = n % kItemQ;
          if (!mbar_wait(&item_empty[slot], ((n / kItemQ) & 1) ^ 1, 34)) {
            ok = false;
            break;
          }
          items[slot] = DecodeItem{seq, ch, grp, L};
          mbar_arrive(&item_full[slot]);
          ++n;
          const int ntok = max(0, min(p.chunk, L - ch * p.chunk));
          const int nb = (ntok + kBox - 1) / kBox;
          const int32_t* bt = p.block_table + static_cast<size_t>(seq) * p.max_pages;
          for (int i = 0; i < 2 * nb; ++i, ++box) {
            const int st = box % p.stages;
            if (!mbar_wait(&empty[st], ((box / p.stages) & 1) ^ 1, 30)) {
              ok = false;
              break;
            }
            const int t0 = ch * p.chunk + (i < nb ? i : i - nb) * kBox;
            const int page = __ldg(bt + t0 / ps);  // t0 < L <= max_pages * page_size
            // An out-of-range page index is reported; TMA fills such a box
            // with zeros instead of reading outside the cache.
            if (i < nb && (page < 0 || page >= p.num_pages)) report_error(7 /* ATTN_ERR_BOUNDS */, seq, page);
            mbar_expect_tx(&full[st], p.stage_bytes);
            tma_load_4d(smem + st * p.stage_bytes, i < nb ? &tmK : &tmV, &full[st], 0, grp * p.hg, t0 % ps, page);
          }
        }
        if (!ok) break;
        if (p.sched == nullptr) break;  // one item per CTA
        const int f = sched_fetch(p.sched, p.sched_tag, owned, U);
        w = f < 0 ? U : static_cast<int>(gridDim.x) + f;
      }
      // A producer that stopped early still makes its final fetch, so that the
      // launch's fetches add up and the counter slot is freed.
      while (p.sched != nullptr && w < U) {
        const int f = sched_fetch(p.sched, p.sched_tag, owned, U);
        w = f < 0 ? U : static_cast<int>(gridDim.x) + f;
      }
      // Terminator for the compute warps.
      const int slot = n % kItemQ;
      if (mbar_wait(&item_empty[slot], ((n / kItemQ) & 1) ^ 1, 35)) {
        items[slot] = DecodeItem{ok ? -1 : -2, 0, 0, 0};
        mbar_arrive(&item_full[slot]);
      }
      // Drain: never leave the CTA with a copy still writing shared memory
      // (after one wait gives up, the rest are not attempted).
      bool drained = true;
      for (int b = max(0, box - p.stages); drained && b < box; ++b)
        drained = mbar_wait(&full[b % p.stages], (b / p.stages) & 1, 31);
    }
    __syncwarp();
  } else if (warp < nw) {
    // ------------------------------------------------------------------ compute warps
    const int kvl = warp / WPH;            // key/value head within the group
    const int qh0 = (warp % WPH) * GW;     // first of this warp's query heads of that kv head
    const int sub = lane % S::LPT;         // 16-byte slice of the key row
    const int grp_l = lane / S::LPT;       // which key row of a pass
    float* sc = scores + warp * p.chunk * GW;  // [token][g] scores, then probabilities
    const uint32_t row_bytes = D * 2;
    const uint32_t slot_stride = p.hg * row_bytes;
    int box = 0;
    for (int n = 0;; ++n) {
      const int islot = n % kItemQ;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&item_full[islot], (n / kItemQ) & 1, 36))) break;
      const DecodeItem it = items[islot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&item_empty[islot]);
      if (it.seq < 0) break;
      const int seq = it.seq, L = it.len;
      const int ntok = max(0, min(p.chunk, L - it.chunk * p.chunk));
      const int nb = (ntok + kBox - 1) / kBox;
      const int nch = L > 0 ? (L + p.chunk - 1) / p.chunk : 1;
      const int kvh = it.group * p.hg + kvl;
      const int head0 = kvh * G + qh0;

      float qf[GW][8];
#pragma unroll
      for (int g = 0; g < GW; ++g) {
        const uint4 wq = __ldg(reinterpret_cast<const uint4*>(p.q + (static_cast<size_t>(seq) * p.Hq + head0 + g) * D +
                                                               sub * 8));
        qf[g][0] = bf16lo(wq.x) * p.scale_log2;
        qf[g][1] = bf16hi(wq.x) * p.scale_log2;
        qf[g][2] = bf16lo(wq.y) * p.scale_log2;
        qf[g][3] = bf16hi(wq.y) * p.scale_log2;
        qf[g][4] = bf16lo(wq.z) * p.scale_log2;
        qf[g][5] = bf16hi(wq.z) * p.scale_log2;
        qf[g][6] = bf16lo(wq.w) * p.scale_log2;
        qf[g][7] = bf16hi(wq.w) * p.scale_log2;
      }

      bool ok = true;
      // ---- K boxes: scores x = (scale log2 e) q . k
      for (int i = 0; ok && i < nb; ++i, ++box) {
        const int st = box % p.stages;
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(&full[st], (box / p.stages) & 1, 32));
        if (!ok) break;
        const uint32_t kb = sbase + st * p.stage_bytes + kvl * row_bytes + sub * 16;
#pragma unroll
        for (int rd = 0; rd < S::PASSES / S::R; ++rd) {
          float part[S::NV];
#pragma unroll
          for (int r = 0; r < S::R; ++r) {
            const int slot = (rd * S::R + r) * S::TPP + grp_l;
            const uint4 wk = ld_shared_v4(kb + slot * slot_stride);
            const float k8[8] = {bf16lo(wk.x), bf16hi(wk.x), bf16lo(wk.y), bf16hi(wk.y),
                                 bf16lo(wk.z), bf16hi(wk.z), bf16lo(wk.w), bf16hi(wk.w)};
#pragma unroll
            for (int g = 0; g < GW; ++g) {
              float a = qf[g][0] * k8[0];
#pragma unroll
              for (int e = 1; e < 8; ++e) a = fmaf(qf[g][e], k8[e], a);
              part[r * GW + g] = a;
            }
          }
          lane_reduce<S::NV, S::LPT, S::SCAT, S::LEVELS>(part, lane);
          const int dup_bits = S::LEVELS - S::SCAT;
          if ((sub & ((1 << dup_bits) - 1)) == 0) {
            const int base = (sub >> dup_bits) * S::KEEP;
#pragma unroll
            for (int v = 0; v < S::KEEP; ++v) {
              const int idx = base + v;
              const int r = idx / GW;
              const int g = idx - r * GW;
              const int slot = (rd * S::R + r) * S::TPP + grp_l;
              sc[(i * kBox + slot) * GW + g] = part[v];
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
      }
      __syncwarp();
      if (!ok) break;

      // ---- softmax over the chunk, per query head g = lane % GW
      float m = -INFINITY;
      float s = 0.f;
      for (int i = lane; i < ntok * GW; i += 32) m = fmaxf(m, sc[i]);
#pragma unroll
      for (int off = GW; off < 32; off <<= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
      for (int i = lane; i < ntok * GW; i += 32) {
        const float e = ex2(sc[i] - m);
        sc[i] = e;
        s += e;
      }
#pragma unroll
      for (int off = GW; off < 32; off <<= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, off);
      __syncwarp();

      // ---- V boxes: o = sum_j p_j v_j
      float acc[GW][8];
#pragma unroll
      for (int g = 0; g < GW; ++g)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[g][e] = 0.f;
      for (int i = 0; ok && i < nb; ++i, ++box) {
        const int st = box % p.stages;
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(&full[st], (box / p.stages) & 1, 33));
        if (!ok) break;
        const uint32_t vb = sbase + st * p.stage_bytes + kvl * row_bytes + sub * 16;
#pragma unroll 4
        for (int pp = 0; pp < S::PASSES; ++pp) {
          const int slot = pp * S::TPP + grp_l;
          const int tok = i * kBox + slot;
          if (tok < ntok) {
            const uint4 wv = ld_shared_v4(vb + slot * slot_stride);
            const float v8[8] = {bf16lo(wv.x), bf16hi(wv.x), bf16lo(wv.y), bf16hi(wv.y),
                                 bf16lo(wv.z), bf16hi(wv.z), bf16lo(wv.w), bf16hi(wv.w)};
            float pg[GW];
#pragma unroll
            for (int g = 0; g < GW; ++g) pg[g] = sc[tok * GW + g];
#pragma unroll
            for (int g = 0; g < GW; ++g)
#pragma unroll
              for (int e = 0; e < 8; ++e) acc[g][e] = fmaf(pg[g], v8[e], acc[g][e]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
      }
      if (!ok) break;

      // rows of a pass were split over lane groups: add them up
#pragma unroll
      for (int off = S::LPT; off < 32; off <<= 1)
#pragma unroll
        for (int g = 0; g < GW; ++g)
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[g][e] += __shfl_xor_sync(0xFFFFFFFFu, acc[g][e], off);
      float mg[GW], sg[GW];
#pragma unroll
      for (int g = 0; g < GW; ++g) {
        mg[g] = __shfl_sync(0xFFFFFFFFu, m, g);
        sg[g] = __shfl_sync(0xFFFFFFFFu, s, g);
      }
      const bool direct = nch <= 1;
      if (grp_l == 0) {
#pragma unroll
        for (int g = 0; g < GW; ++g) {
          const int head = head0 + g;
          const bool any = ntok > 0 && sg[g] > 0.f;
          const float inv = any ? 1.f / sg[g] : 0.f;
          const float lse_v = any ? (mg[g] + lg2(sg[g])) * 0.69314718055994531f : -INFINITY;
          float ov[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) ov[e] = acc[g][e] * inv;
          if (direct) {
            const size_t off = (static_cast<size_t>(seq) * p.Hq + head) * D + sub * 8;
            if (p.o_f32) {
              float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + off);
              dst[0] = make_float4(ov[0], ov[1], ov[2], ov[3]);
              dst[1] = make_float4(ov[4], ov[5], ov[6], ov[7]);
            } else {
              *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + off) =
                  make_uint4(pack_bf16(ov[0], ov[1]), pack_bf16(ov[2], ov[3]), pack_bf16(ov[4], ov[5]),
                             pack_bf16(ov[6], ov[7]));
            }
            if (sub == 0) p.lse[static_cast<size_t>(seq) * p.Hq + head] = lse_v;
          } else {
            const size_t row = (static_cast<size_t>(seq) * p.n_splits + it.chunk) * p.Hq + head;
            float4* dst = reinterpret_cast<float4*>(p.ws_o + row * D + sub * 8);
            dst[0] = make_float4(ov[0], ov[1], ov[2], ov[3]);
            dst[1] = make_float4(ov[4], ov[5], ov[6], ov[7]);
            if (sub == 0) p.ws_lse[row] = lse_v;
          }
        }
      }
      if (!direct) {
        // Publish this chunk's partial rows (every lane fences its own
        // writes), then count the arrival; the arrival that completes the
        // sequence merges this warp's heads.
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0) {
          unsigned long long* cnt = p.ws_cnt + (static_cast<size_t>(seq) * p.ngroups + it.group) * nw + warp;
          last = merge_arrive(cnt, p.epoch, nch) ? 1 : 0;
        }
        last = __shfl_sync(0xFFFFFFFFu, last, 0);
        if (last) {
          __threadfence();
          merge_heads<D, GW>(p, seq, head0, nch, lane);
        }
      }
    }
  }
}

}  // namespace attn
