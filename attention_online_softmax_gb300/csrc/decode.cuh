// Paged split-KV decode for sm_103a: one query row per (sequence, query head)
// against a paged KV cache, as a bandwidth-bound GEMV-class stage.
//
// decode_split_kernel: one CTA per (sequence, key chunk, group of hg key/value
// heads).  A producer thread streams the chunk's cached tokens with TMA in
// boxes of [16 slots][hg heads][d] -- first the K boxes, then the V boxes --
// into a ring of shared-memory stages, so every global read is a run of d*2
// contiguous bytes per (slot, head); for page sizes above 16 a box is the
// 16-slot window of a page at the token's slot offset.  Compute warp w serves
// key/value head w / WPH of the group and GW of the query heads that share it
// (grouped-query attention: one read of K/V serves the whole group; a group
// of 16 query heads is split over two warps).  Lanes own 16-byte slices of a
// key row; partial dot products are reduced across the lanes of a row by a
// reduce-scatter over shuffles.  The chunk's scores stay in shared memory, so
// the chunk is softmaxed once (max, 2^(x - m), sum) and then the V boxes are
// accumulated.  The chunk's partial state is stored as (O_c, lse_c) =
// (o / l, m + ln l) ("online softmax as a monoid", Tang abstract).
//
// decode_combine_kernel: merges the chunk partials of each (sequence, head):
// LSE = logsumexp_c(lse_c), O = sum_c exp(lse_c - LSE) O_c -- the merge of
// partial states of the block recurrence in "Compilers and Kernels", section
// "FlashAttention changes the algorithm around IO", applied to whole chunks.
// It is launched as a programmatic dependent of the split kernel, so its
// launch overlaps the split kernel's tail.  Sequences that fit one chunk are
// finished by the split kernel directly.
#pragma once

#include "ptx.cuh"

namespace attn {

constexpr int kBox = 16;         // cached tokens per TMA box (one ring stage)
constexpr int kChunkMax = 256;   // tokens per split, upper bound
constexpr int kMaxStages = 8;

struct DecodeParams {
  const uint16_t* q;
  const int32_t* block_table;
  const int32_t* seqlens;
  void* o;
  float* lse;
  float* ws_o;    // [num_seqs][n_splits][Hq][D] chunk outputs O_c
  float* ws_lse;  // [num_seqs][n_splits][Hq]    chunk lse_c
  int num_seqs, Hq, Hkv, num_pages, max_pages, max_seqlen, page_size;
  int chunk;      // tokens per split: multiple of 16, <= kChunkMax
  int n_splits;   // ceil(max_seqlen / chunk), >= 1
  int hg;         // key/value heads per CTA
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

// Up to four query heads per warp and d <= 128: two CTAs per SM (registers capped for it).
template <int D, int GW, int WPH>
__global__ void __launch_bounds__(288, (GW <= 4 && D <= 128) ? 2 : 1)
    decode_split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                        const DecodeParams p) {
  using S = DecodeShape<D, GW>;
  constexpr int G = GW * WPH;  // query heads per key/value head
  const int split = static_cast<int>(blockIdx.x % p.n_splits);
  const int seq = static_cast<int>(blockIdx.x / p.n_splits);
  const int L = decode_len(p, seq, split == 0 && blockIdx.y == 0);
  const int t_begin = split * p.chunk;
  if (t_begin >= L && split > 0) return;  // empty chunk (uniform for the CTA)
  const int ntok = min(L - t_begin, p.chunk) > 0 ? min(L - t_begin, p.chunk) : 0;
  const int nbox = (ntok + kBox - 1) / kBox;
  const int n_split_seq = L > 0 ? (L + p.chunk - 1) / p.chunk : 1;
  const int hg = p.hg;
  const int nw = hg * WPH;  // compute warps
  const int kvh0 = blockIdx.y * hg;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const uint32_t sbase = smem_u32(smem);
  float* scores = reinterpret_cast<float*>(smem + p.stages * p.stage_bytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.stages * p.stage_bytes + nw * p.chunk * GW * 4);
  uint64_t* empty = full + kMaxStages;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], nw);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == nw) {
    // ------------------------------------------------------------------ producer
    if (lane == 0 && nbox > 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const int ps = p.page_size;
      const int32_t* bt = p.block_table + static_cast<size_t>(seq) * p.max_pages;
      int issued = 0;
      for (int item = 0; item < 2 * nbox; ++item) {
        const int st = item % p.stages;
        const uint32_t ph = (item / p.stages) & 1;
        if (!mbar_wait(&empty[st], ph ^ 1, 30)) break;
        const int t0 = t_begin + (item < nbox ? item : item - nbox) * kBox;
        const int page = __ldg(bt + t0 / ps);  // t0 < L <= max_pages * page_size
        // An out-of-range page index is reported; TMA fills such a box with
        // zeros instead of reading outside the cache.
        if (item < nbox && (page < 0 || page >= p.num_pages)) report_error(7 /* ATTN_ERR_BOUNDS */, seq, page);
        mbar_expect_tx(&full[st], p.stage_bytes);
        tma_load_4d(smem + st * p.stage_bytes, item < nbox ? &tmK : &tmV, &full[st], 0, kvh0, t0 % ps, page);
        issued = item + 1;
      }
      // Drain: never leave the CTA with a copy still writing shared memory
      // (after one wait gives up, the rest are not attempted).
      bool drained = true;
      for (int item = max(0, issued - p.stages); drained && item < issued; ++item)
        drained = mbar_wait(&full[item % p.stages], (item / p.stages) & 1, 31);
    }
    __syncwarp();
  } else if (warp < nw) {
    // ------------------------------------------------------------------ compute warps
    const int hl = warp / WPH;           // key/value head within the group
    const int kvh = kvh0 + hl;
    const int head0 = kvh * G + (warp % WPH) * GW;  // first of this warp's query heads
    const int sub = lane % S::LPT;       // 16-byte slice of the key row
    const int grp = lane / S::LPT;       // which key row of a pass
    float* sc = scores + warp * p.chunk * GW;  // [token][g] scores, then probabilities
    const uint32_t row_bytes = D * 2;
    const uint32_t slot_stride = hg * row_bytes;

    float qf[GW][8];
#pragma unroll
    for (int g = 0; g < GW; ++g) {
      const uint4 w = *reinterpret_cast<const uint4*>(
          p.q + (static_cast<size_t>(seq) * p.Hq + head0 + g) * D + sub * 8);
      qf[g][0] = bf16lo(w.x) * p.scale_log2;
      qf[g][1] = bf16hi(w.x) * p.scale_log2;
      qf[g][2] = bf16lo(w.y) * p.scale_log2;
      qf[g][3] = bf16hi(w.y) * p.scale_log2;
      qf[g][4] = bf16lo(w.z) * p.scale_log2;
      qf[g][5] = bf16hi(w.z) * p.scale_log2;
      qf[g][6] = bf16lo(w.w) * p.scale_log2;
      qf[g][7] = bf16hi(w.w) * p.scale_log2;
    }

    bool ok = true;
    // ---- K boxes: scores x = (scale log2 e) q . k
    for (int i = 0; ok && i < nbox; ++i) {
      const int st = i % p.stages;
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(&full[st], (i / p.stages) & 1, 32));
      if (!ok) break;
      const uint32_t kb = sbase + st * p.stage_bytes + hl * row_bytes + sub * 16;
#pragma unroll
      for (int rd = 0; rd < S::PASSES / S::R; ++rd) {
        float part[S::NV];
#pragma unroll
        for (int r = 0; r < S::R; ++r) {
          const int slot = (rd * S::R + r) * S::TPP + grp;
          const uint4 w = ld_shared_v4(kb + slot * slot_stride);
          const float k8[8] = {bf16lo(w.x), bf16hi(w.x), bf16lo(w.y), bf16hi(w.y),
                               bf16lo(w.z), bf16hi(w.z), bf16lo(w.w), bf16hi(w.w)};
          if constexpr (GW == 1) {
            float a = qf[0][0] * k8[0];
#pragma unroll
            for (int e = 1; e < 8; ++e) a = fmaf(qf[0][e], k8[e], a);
            part[r] = a;
          } else {
            // Two query heads per paired f32x2 multiply-add (the same
            // operations, in the same order, as one head at a time).
#pragma unroll
            for (int g = 0; g < GW; g += 2) {
              float a0, a1;
              fmul2(a0, a1, qf[g][0], qf[g + 1][0], k8[0], k8[0]);
#pragma unroll
              for (int e = 1; e < 8; ++e) ffma2(a0, a1, qf[g][e], qf[g + 1][e], k8[e], k8[e], a0, a1);
              part[r * GW + g] = a0;
              part[r * GW + g + 1] = a1;
            }
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
            const int slot = (rd * S::R + r) * S::TPP + grp;
            sc[(i * kBox + slot) * GW + g] = part[v];
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    __syncwarp();

    // ---- softmax over the chunk, per query head g = lane % GW
    float m = -INFINITY;
    float s = 0.f;
    if (ok) {
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
    }
    __syncwarp();

    // ---- V boxes: o = sum_j p_j v_j
    float acc[GW][8];
#pragma unroll
    for (int g = 0; g < GW; ++g)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[g][e] = 0.f;
    for (int i = 0; ok && i < nbox; ++i) {
      const int item = nbox + i;
      const int st = item % p.stages;
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(&full[st], (item / p.stages) & 1, 33));
      if (!ok) break;
      const uint32_t vb = sbase + st * p.stage_bytes + hl * row_bytes + sub * 16;
#pragma unroll 4
      for (int ps = 0; ps < S::PASSES; ++ps) {
        const int slot = ps * S::TPP + grp;
        const int tok = i * kBox + slot;
        if (tok < ntok) {
          const uint4 w = ld_shared_v4(vb + slot * slot_stride);
          const float v8[8] = {bf16lo(w.x), bf16hi(w.x), bf16lo(w.y), bf16hi(w.y),
                               bf16lo(w.z), bf16hi(w.z), bf16lo(w.w), bf16hi(w.w)};
          float pg[GW];
#pragma unroll
          for (int g = 0; g < GW; ++g) pg[g] = sc[tok * GW + g];
#pragma unroll
          for (int g = 0; g < GW; ++g)
#pragma unroll
            for (int e = 0; e < 8; e += 2)
              ffma2(acc[g][e], acc[g][e + 1], pg[g], pg[g], v8[e], v8[e + 1], acc[g][e], acc[g][e + 1]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }

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

    if (ok && grp == 0) {
      const bool direct = n_split_seq <= 1;
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
          const size_t row = (static_cast<size_t>(seq) * p.n_splits + split) * p.Hq + head;
          float4* dst = reinterpret_cast<float4*>(p.ws_o + row * D + sub * 8);
          dst[0] = make_float4(ov[0], ov[1], ov[2], ov[3]);
          dst[1] = make_float4(ov[4], ov[5], ov[6], ov[7]);
          if (sub == 0) p.ws_lse[row] = lse_v;
        }
      }
    }
  }
  __syncthreads();
  // This CTA's partials are written: the combine kernel (launched as a
  // programmatic dependent) may start once every CTA got here.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// One block of 4 warps per (sequence, query head); lanes own D/32 consecutive
// elements.  Launched as a programmatic dependent of the split kernel: it
// waits on the grid dependency before reading any partial.  Every warp takes
// the maximum of the chunk lse values; warp w then takes chunks w, w + 4,
// ..., eight rows in flight at a time, and the four partial sums meet in
// shared memory.
template <int D>
__global__ void __launch_bounds__(128) decode_combine_kernel(const DecodeParams p) {
  constexpr int E = D / 32;
  constexpr int kRows = 8;  // chunk rows in flight per warp
  __shared__ float s_acc[4][D];
  __shared__ float s_w[4];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int seq = blockIdx.x;
  const int head = blockIdx.y;
  const int L = decode_len(p, seq, false);
  const int ns = L > 0 ? (L + p.chunk - 1) / p.chunk : 1;
  if (ns <= 1) return;  // finished by the split kernel (uniform for the block)
  const size_t row0 = static_cast<size_t>(seq) * p.n_splits * p.Hq + head;
  float m = -INFINITY;
  for (int c = lane; c < ns; c += 32) m = fmaxf(m, p.ws_lse[row0 + static_cast<size_t>(c) * p.Hq]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float wsum = 0.f;  // the same in every lane
  for (int c0 = warp; c0 < ns; c0 += 4 * kRows) {
    float v[kRows][E];
    float lc[kRows];
#pragma unroll
    for (int u = 0; u < kRows; ++u) {
      const int c = min(c0 + 4 * u, ns - 1);  // in range; weight 0 past the end
      const size_t r = row0 + static_cast<size_t>(c) * p.Hq;
      lc[u] = p.ws_lse[r];
      const float* src = p.ws_o + r * D + lane * E;
#pragma unroll
      for (int e = 0; e < E; e += 2) {
        const float2 x = *reinterpret_cast<const float2*>(src + e);
        v[u][e] = x.x;
        v[u][e + 1] = x.y;
      }
    }
#pragma unroll
    for (int u = 0; u < kRows; ++u) {
      const float w = c0 + 4 * u < ns ? ex2((lc[u] - m) * 1.4426950408889634f) : 0.f;
      wsum += w;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = fmaf(w, v[u][e], acc[e]);
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) s_acc[warp][lane * E + e] = acc[e];
  if (lane == 0) s_w[warp] = wsum;
  __syncthreads();
  if (warp != 0) return;
  const float wt = s_w[0] + s_w[1] + s_w[2] + s_w[3];
  const float inv = 1.f / wt;
  float o[E];
#pragma unroll
  for (int e = 0; e < E; ++e)
    o[e] = (s_acc[0][lane * E + e] + s_acc[1][lane * E + e] + s_acc[2][lane * E + e] + s_acc[3][lane * E + e]) * inv;
  const size_t off = (static_cast<size_t>(seq) * p.Hq + head) * D + lane * E;
  if (p.o_f32) {
    float* dst = static_cast<float*>(p.o) + off;
#pragma unroll
    for (int e = 0; e < E; e += 2) *reinterpret_cast<float2*>(dst + e) = make_float2(o[e], o[e + 1]);
  } else {
    uint32_t* dst = reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(p.o) + off);
#pragma unroll
    for (int e = 0; e < E; e += 2) dst[e / 2] = pack_bf16(o[e], o[e + 1]);
  }
  if (lane == 0) p.lse[static_cast<size_t>(seq) * p.Hq + head] = m + logf(wt);
}

}  // namespace attn
