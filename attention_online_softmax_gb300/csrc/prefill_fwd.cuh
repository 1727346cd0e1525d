// Fused attention forward (prefill) for sm_103a.
//
// A persistent kernel: one CTA per SM takes work units from a per-launch
// atomic counter until none are left.  A unit is NQ 128-row query tiles
// (NQ = 2 for d <= 128 when that still gives two units per SM, else 1) of one
// (batch, query head) -- or, in the PAGED variant, of one sequence and query
// head of a chunked prefill against a paged KV cache -- computed
// against the key/value tiles those rows may see with the block recurrence of
// "Compilers and Kernels", section "FlashAttention changes the algorithm
// around IO": for each key block B_t the row state (m, l, o) is updated by
//     m_t = max(m_{t-1}, b_t),  alpha_t = exp(m_{t-1} - m_t),
//     l_t = alpha_t l_{t-1} + sum exp(S - m_t),  o_t = alpha_t o_{t-1} + sum exp(S - m_t) v,
// and O = o_T / l_T, LSE = m_T + ln l_T at the end.  Scores never leave the SM.
// Units are handed out longest causal unit first within groups of heads, so
// the uneven causal units pack well while each group's K/V stays in L2.
//
// Roles (64 + 128*NQ threads, plus a bias-loader warp for a staged dense bias,
// a second MMA-issuing warp with separate P slots, and a second producer warp
// for the paged cache):
//   warp 0        TMA producer: takes the next unit from the work counter and
//                 passes it to the other roles through a small shared-memory
//                 queue, loads the unit's NQ query tiles, then its K_t, V_t
//                 tiles (shared by all query tiles of the unit) into a
//                 STAGES-deep shared-memory ring (128-byte swizzle) that runs on
//                 across units, so the next unit's loads overlap this one's end.
//   warp 1        allocates tensor memory once; one thread issues tcgen05.mma:
//                 S_j = Q_j K_t^T (smem x smem) into TMEM, then
//                 O_j += P_j V_t with P_j read from TMEM (tmem x smem).
//   warps 2..     one softmax warpgroup per query tile, one thread per row:
//                 reads S from TMEM, adds the bias terms and applies the masks,
//                 updates the running max, writes P = 2^(x - m) as bf16 to
//                 TMEM, rescales O in TMEM when the max moved, and writes O / l
//                 and LSE.
//
// Tensor memory (512 columns): O_j at columns [j*D, (j+1)*D); two S slots of
// 128 columns after them.  With NQ = 2 slot j belongs to query tile j and the
// MMA order PV_A(t-1), S_A(t), PV_B(t-1), S_B(t) lets one warpgroup's softmax
// overlap the other tile's MMAs.  With NQ = 1 the slots alternate over key
// tiles: S(t+1) is computed while tile t is softmaxed.  P (bf16, 64 columns)
// overwrites the first half of its S slot; tcgen05 MMAs from one thread run in
// issue order, so the next S into that slot is issued after the P V product.
// The plain kernel with NQ = 1 and d <= 128 instead keeps P in two slots of
// its own after the S slots (O + 2 S + 2 P = 512 columns at d = 128): S(t+2)
// is issued once the softmax has read S(t), and a second thread issues the
// P V products.
// A unit's first P V product overwrites O_j only after the previous unit's
// epilogue has read it (barrier o_free).  Barrier phases run on across units.
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

namespace attn {

constexpr int kBM = 128;  // query rows per tile (TMEM lanes)
constexpr int kBN = 128;  // keys per tile
constexpr float kRescaleLog2 = 8.0f;
constexpr int kUnitQ = 4;  // depth of the in-CTA queue of fetched units
// Ring of per-step K/V barriers (plain kernel, two query tiles): more entries
// than any producer lead over the MMA thread, so phases never alias.
constexpr int kStepR = 16;

struct PrefillParams {
  void* o;
  float* lse;
  unsigned long long* sched;  // this launch's counter slot: (owner tag << 32) | fetches; 0 when free
  unsigned sched_tag;         // this launch's nonzero owner tag
  int B, Hq, Hkv, Nq, Nk;
  int causal;
  int o_f32;
  int n_units;       // units per (batch, head): ceil(Nq / (128 * NQ))
  int group;         // (batch, head) pairs scheduled together, longest units first
  float scale_log2;  // scale * log2(e), > 0
  // Additive bias C beyond the causal mask (all off in the plain call):
  int window;                 // > 0: key j allowed only if j > i + (Nk - Nq) - window
  const float* alibi;         // null or [Hq]: adds alibi[h] * (j - i - (Nk - Nq))
  const uint16_t* bias;       // null or bf16 bias[b*bias_sb + h*bias_sh + i*Nk + j]
  long long bias_sb, bias_sh;
  int bias_hmul, bias_bmul;   // staged bias: head / batch coordinate multipliers (0: broadcast)
  // Chunked prefill against a paged KV cache (PAGED kernels only): sequence s
  // owns packed query tokens [cu_q[s], cu_q[s+1]), the last ones of a context
  // of seqlens_k[s] tokens whose key t sits in page block_table[s][t / page_size].
  const int32_t* cu_q;
  const int32_t* seqlens_k;
  const int32_t* block_table;
  const int32_t* unit_prefix;  // [num_seqs + 1] units before each rank of seq_order (plan kernel)
  const int32_t* seq_order;    // [num_seqs] sequences in dispatch order, longest context first (plan kernel)
  int num_seqs, max_pages, page_size, num_pages;
};


template <int D, int NQ, int STAGES, int BSLOTS = 0, bool PSEP = false, int PW = 1>
struct PrefillLayout {
  // warp 0 TMA producer, warp 1 MMA issuer, 4 softmax warps per query tile,
  // and with a staged bias one more warp that loads the bias tiles.
  // Separate P slots (PSEP, one query tile, d <= 128): a second MMA-issuing
  // warp takes the P V products.  PW = 2 (paged cache): a second producer
  // warp, the last one, issues half of each item's page boxes.
  static constexpr bool kPSep = PSEP && NQ == 1 && D <= 128;
  static constexpr bool kSplit = kPSep;
  static constexpr int kPVWarp = 2 + 4 * NQ + (BSLOTS > 0 ? 1 : 0);
  static constexpr int kProd2Warp = 2 + 4 * NQ + (BSLOTS > 0 ? 1 : 0) + (kSplit ? 1 : 0);
  static constexpr int kThreads = 64 + 128 * NQ + (BSLOTS > 0 ? 32 : 0) + (kSplit ? 32 : 0) + (PW - 1) * 32;
  static constexpr int kQBytes = kBM * D * 2;
  // K and V tiles stream in items of up to 128 head-dim columns (kH items per
  // tile), so with d = 256 a 64 KB tile occupies two 32 KB ring stages and
  // loading the next tile overlaps the current one's MMAs.
  static constexpr int kDI = D < 128 ? D : 128;  // head-dim columns per item
  static constexpr int kH = D / kDI;             // items per K (or V) tile
  static constexpr int kKVBytes = kBN * kDI * 2; // one ring stage
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = kQOff + NQ * kQBytes;
  // Staged dense bias: BSLOTS slots of one 128 x 128 bf16 tile each, as two
  // 128-byte-swizzled [128 rows][64 keys] boxes.
  static constexpr int kBiasBytes = kBM * kBN * 2;
  static constexpr int kBiasOff = kKVOff + STAGES * kKVBytes;
  static constexpr int kBarOff = kBiasOff + BSLOTS * kBiasBytes;
  // q_full, q_empty, kv_full[S], kv_empty[S], s_full[2], p_full[2], pv_done,
  // (s_free[2], pv_free[2], step_full[kStepR], step_empty[kStepR] after tail_bar),
  // o_done[2], o_free[2], unit_full[Q], unit_empty[Q], mma_drain,
  // bias_full[BSLOTS], bias_empty[BSLOTS], tail_bar[2]
  static constexpr int kNumBars = 2 + 2 * STAGES + 2 + 2 + 1 + 2 + 2 + 2 * kUnitQ + 1 + 2 * BSLOTS + 2 + 4 + 2 * kStepR;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // tmem slot, unit queue
  static constexpr int kUnitBytes = 64;                      // one decoded unit in the queue
  static constexpr int kBytes = kMiscOff + 16 + kUnitBytes * kUnitQ;
  // Dynamic shared memory requested: at least 115 KB so that no second CTA
  // (which would wait for this one's tensor memory) shares the SM.
  static constexpr int kAlloc = (kBytes + 1024) > 117760 ? (kBytes + 1024) : 117760;
  static constexpr int kTmemCols = 512;
  static constexpr int kSCol = NQ * D;          // first S slot column
  // One query tile and d <= 128: P gets its own two 64-column slots after the
  // S slots, so the next S products need not wait for the P V products.
  static constexpr int kPCol = kSCol + 2 * kBN;
  static_assert(!kPSep || kPCol + kBN <= 512, "tensor memory for separate P slots");
  static_assert(NQ * D + 2 * kBN <= kTmemCols, "tensor memory budget");
  static_assert(kAlloc <= 232448, "shared memory budget");
  static_assert(D % 64 == 0, "head dim");
  static_assert(NQ == 1 || NQ == 2, "query tiles per CTA");
};

// Position of K(t) / V(t) in a unit's load order, in tile items (each of
// kH ring stages).  With two query tiles the MMA thread consumes K(t), V(t),
// K(t+1), ... in that order; with one query tile it computes S(t+1) before
// P V(t), so it consumes K(0), K(1), V(0), K(2), V(1), ..., V(T-1) -- and the
// producer loads in the same order, so the ring drains first in, first out.
//
// With separate P slots (PSEP) the MMA thread issues S(t+2) before P V(t):
// K(0), K(1), then K(t+2), V(t) for t = 0 .. T-3, then V(T-2), V(T-1).
template <int NQ, bool PSEP = false>
__device__ __forceinline__ int k_pos(int t) {
  if (PSEP) return t < 2 ? t : 2 * t - 2;
  return NQ == 2 ? 2 * t : (t == 0 ? 0 : 2 * t - 1);
}
template <int NQ, bool PSEP = false>
__device__ __forceinline__ int v_pos(int t, int T) {
  if (PSEP) return T == 1 ? 1 : (t <= T - 3 ? 2 * t + 3 : T + t);
  return NQ == 2 ? 2 * t + 1 : (t == T - 1 ? 2 * T - 1 : 2 * t + 2);
}

// One work unit: its (batch, head) and first query row, and the key tiles each
// of its query tiles needs (0 for a tile past Nq or fully masked).
template <int NQ>
struct Unit {
  int idx;               // position in the launch's unit order (-1: no work left, -2: timed out)
  int bh, kvh, q0;       // (batch, head) row block (paged: the query head), its KV head, first query row
  int tmin, T;           // key tiles loaded: [tmin, tmin + T)
  int lo[NQ], hi[NQ];    // key tiles each query tile needs: [lo, hi), empty if lo >= hi
  int nq, nk, qbase, seq;  // this problem's query and key counts, first packed query token, sequence
};

// Unit `idx`.  Plain: the grouped longest-first order over (batch, head,
// query-tile) (0 <= idx < B*Hq*n_units).  Paged: sequence by sequence in the
// plan kernel's order (longest context first; unit prefix sums over that
// order), within a sequence its last query tile first, heads fastest.
template <int NQ, bool PAGED>
__device__ __forceinline__ Unit<NQ> unit_of(const PrefillParams& p, int idx) {
  Unit<NQ> u;
  u.idx = idx;
  if (PAGED) {
    int a = 0, b = p.num_seqs - 1;  // last rank whose first unit is <= idx
    while (a < b) {
      const int mid = (a + b + 1) >> 1;
      if (__ldg(p.unit_prefix + mid) <= idx) a = mid;
      else b = mid - 1;
    }
    const int local = idx - __ldg(p.unit_prefix + a);
    const int s = __ldg(p.seq_order + a);
    u.seq = s;
    u.qbase = __ldg(p.cu_q + s);
    u.nq = __ldg(p.cu_q + s + 1) - u.qbase;
    u.nk = __ldg(p.seqlens_k + s);
    const int ntiles = (u.nq + kBM * NQ - 1) / (kBM * NQ);  // units of NQ query tiles
    u.bh = local % p.Hq;
    u.kvh = u.bh / (p.Hq / p.Hkv);
    u.q0 = (ntiles - 1 - local / p.Hq) * (kBM * NQ);
  } else {
    const int BH = p.B * p.Hq;
    const int per_group = p.group * p.n_units;
    const int grp = idx / per_group;
    const int in = idx - grp * per_group;
    const int gsize = min(p.group, BH - grp * p.group);
    const int rank = in / gsize;
    u.bh = grp * p.group + (in - rank * gsize);
    const int un = p.n_units - 1 - rank;
    const int b = u.bh / p.Hq;
    const int h = u.bh - b * p.Hq;
    u.kvh = b * p.Hkv + h / (p.Hq / p.Hkv);
    u.q0 = un * (kBM * NQ);
    u.nq = p.Nq;
    u.nk = p.Nk;
    u.qbase = 0;
    u.seq = 0;
  }
  const int diag = u.nk - u.nq;
  int tmax = 0;
  u.tmin = 0x7FFFFFFF;
#pragma unroll
  for (int j = 0; j < NQ; ++j) {
    const int r0 = u.q0 + j * kBM;
    int kbeg = 0, kend = 0;  // keys [kbeg, kend) some row of the tile may see
    if (r0 < u.nq) {
      kend = u.nk;
      if (p.causal) kend = max(0, min(u.nk, min(r0 + kBM, u.nq) - 1 + diag + 1));
      if (p.window > 0) kbeg = max(0, r0 + diag - p.window + 1);
    }
    u.lo[j] = kbeg / kBN;
    u.hi[j] = kend > kbeg ? (kend + kBN - 1) / kBN : u.lo[j];
    if (u.hi[j] > u.lo[j]) {
      u.tmin = min(u.tmin, u.lo[j]);
      tmax = max(tmax, u.hi[j]);
    }
  }
  if (tmax == 0) u.tmin = 0;
  u.T = tmax - u.tmin;
  return u;
}

// Item i of a unit's K/V load order (kH items per tile): its key tile t
// (relative to the unit's first), kind (0: K, 1: V) and head-dim part hh.
template <int NQ, int KH, bool PSEP = false>
__device__ __forceinline__ void load_item(int i, int T, int& t, int& kind, int& hh) {
  const int pos = i / KH;
  hh = i % KH;
  if (PSEP) {
    if (T == 1) {
      t = 0;
      kind = pos;
    } else if (pos < 2) {
      t = pos;
      kind = 0;
    } else if (pos - 2 < 2 * (T - 2)) {
      const int q = pos - 2;
      kind = q & 1;                      // even: K(q/2 + 2), odd: V(q/2)
      t = (q >> 1) + (kind == 0 ? 2 : 0);
    } else {
      t = T - 2 + (pos - 2 - 2 * (T - 2));
      kind = 1;
    }
  } else if (NQ == 2) {
    t = pos >> 1;
    kind = pos & 1;
  } else if (pos == 0) {
    t = 0;
    kind = 0;
  } else if (pos == 2 * T - 1) {
    t = T - 1;
    kind = 1;
  } else {
    kind = (pos & 1) ? 0 : 1;  // odd: K((pos+1)/2), even: V(pos/2 - 1)
    t = kind == 0 ? (pos + 1) >> 1 : (pos >> 1) - 1;
  }
}

// BIAS: 0 no additive bias beyond causal / window masks; 1 ALiBi slopes and/or
// a dense bias read by the softmax threads from global memory; 2 the dense
// bias staged tile by tile into shared memory by the producer (tmB).
template <int BIAS>
__host__ __device__ constexpr int bias_slots() { return BIAS == 2 ? 2 : 0; }
template <int BIAS>
__host__ __device__ constexpr int bias_ring() { return BIAS == 2 ? 2 : 1; }  // modulus (never 0)

// PAGED: Q, O and LSE packed over the sequences' tokens ([total_q][Hq][d],
// [total_q][Hq]); K and V read page by page from the paged cache (tmK, tmV
// box one page of one KV head); tmB is unused.
// Separate P slots and split MMA issue pay off for the plain kernel (measured:
// +9% at B1 H16 N2048 d128); the additive-bias and paged variants, whose
// softmax or producer warps are busier, measured slower with them and keep
// P in the S slot with one MMA-issuing thread.
template <int BIAS, bool PAGED>
__host__ __device__ constexpr bool psep_path() { return BIAS == 0 && !PAGED; }
// Producer warps: two for the paged cache, whose key tile is up to 16 page
// boxes per item (a warp hands its lanes' TMA copies over one at a time, at
// ~60-80 cycles each), one otherwise.
template <bool PAGED>
__host__ __device__ constexpr int producer_warps() { return PAGED ? 2 : 1; }

template <int D, int NQ, int STAGES, int BIAS, bool PAGED = false>
__global__ void __launch_bounds__(
    PrefillLayout<D, NQ, STAGES, bias_slots<BIAS>(), psep_path<BIAS, PAGED>(), producer_warps<PAGED>()>::kThreads, 1)
    prefill_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmB,
                       const PrefillParams p) {
  using L = PrefillLayout<D, NQ, STAGES, bias_slots<BIAS>(), psep_path<BIAS, PAGED>(), producer_warps<PAGED>()>;
  static_assert(BIAS == 0 || NQ == 1, "additive-bias variants run one query tile per unit");
  // With ALiBi slopes a unit's key tiles are taken from the last to the
  // first: the ALiBi term grows with the key index, so the row maxima are
  // met on the first tile taken and O seldom needs rescaling afterwards
  // (the block recurrence gives the same result in any tile order, up to
  // the rounding of P against a different reference maximum).
  const bool rev_tiles = BIAS != 0 && p.alibi != nullptr;
  static_assert(!PAGED || BIAS == 0, "paged prefill: no dense bias");
  static_assert(sizeof(Unit<NQ>) <= L::kUnitBytes, "unit queue entry");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const uint32_t sbase = smem_u32(smem);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* q_full = bars;
  uint64_t* q_empty = bars + 1;
  uint64_t* kv_full = bars + 2;
  uint64_t* kv_empty = kv_full + STAGES;
  uint64_t* s_full = kv_empty + STAGES;
  uint64_t* p_full = s_full + 2;
  uint64_t* pv_done = p_full + 2;
  uint64_t* o_done = pv_done + 1;
  uint64_t* o_free = o_done + 2;
  uint64_t* unit_full = o_free + 2;
  uint64_t* unit_empty = unit_full + kUnitQ;
  uint64_t* mma_drain = unit_empty + kUnitQ;
  uint64_t* bias_full = mma_drain + 1;
  uint64_t* bias_empty = bias_full + bias_slots<BIAS>();
  uint64_t* tail_bar = bias_empty + bias_slots<BIAS>();  // [2] paged: a partly filled value page, per producer warp
  uint64_t* s_free = tail_bar + 2;   // [2] separate P slots: the softmax has read S from this slot
  uint64_t* pv_free = s_free + 2;    // [2] separate P slots: the P V product of this P slot is complete
  uint64_t* step_full = pv_free + 2;         // [kStepR] step ring: V(t-1) and K(t) have landed
  uint64_t* step_empty = step_full + kStepR;  // [kStepR] step ring: the step's products are done with them
  // Plain kernel with two query tiles: the K/V ring is gated per MMA step
  // (V(t-1) and K(t), consecutive items) rather than per item -- one barrier
  // wait and one commit per step for the issuing thread instead of two each.
  constexpr bool kStepRing = NQ == 2;
  static_assert(!kStepRing || L::kH == 1, "step ring: one item per K or V tile");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  Unit<NQ>* unit_q = reinterpret_cast<Unit<NQ>*>(smem + L::kMiscOff + 16);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (PAGED) {
    // Value rows past a sequence's context are never loaded, so every K/V
    // ring byte the MMAs read is a real cache row or this zero: no NaN from an
    // unused cache slot can reach O through a zero weight.
    for (int i = threadIdx.x; i < STAGES * L::kKVBytes / 16; i += blockDim.x)
      st_shared_v4(sbase + L::kKVOff + i * 16, 0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
  }

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&kv_full[s], producer_warps<PAGED>());  // one arrival per producer warp
      mbar_init(&kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 4);
      mbar_init(&o_done[i], 1);
      mbar_init(&o_free[i], 4);
    }
    for (int i = 0; i < kUnitQ; ++i) {
      mbar_init(&unit_full[i], 1);
      // MMA thread + lane 0 of every softmax warp (+ the bias loader, the
      // second MMA-issuing warp, the second producer warp)
      mbar_init(&unit_empty[i],
                1 + 4 * NQ + (BIAS == 2 ? 1 : 0) + (L::kSplit ? 1 : 0) + (producer_warps<PAGED>() - 1));
    }
    mbar_init(pv_done, 1);
    mbar_init(mma_drain, L::kSplit ? 2 : 1);  // one commit per MMA-issuing thread
    mbar_init(&tail_bar[0], 1);
    mbar_init(&tail_bar[1], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_free[i], 4);
      mbar_init(&pv_free[i], 1);
    }
    for (int i = 0; i < kStepR; ++i) {
      mbar_init(&step_full[i], producer_warps<PAGED>());
      mbar_init(&step_empty[i], 1);
    }
    for (int i = 0; i < bias_slots<BIAS>(); ++i) {
      mbar_init(&bias_full[i], 1);
      mbar_init(&bias_empty[i], 4);  // lane 0 of every softmax warp
    }
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

  // Consumers' view of the unit queue: the n-th unit this CTA processes
  // (idx -1: no work left, -2: the wait timed out).  The entry is copied out
  // before the caller releases the slot.
  auto next_unit = [&](int n, int where) -> Unit<NQ> {
    const int slot = n % kUnitQ;
    Unit<NQ> u;
    if (!mbar_wait(&unit_full[slot], (n / kUnitQ) & 1, where)) {
      u.idx = -2;
      return u;
    }
    u = unit_q[slot];
    return u;
  };

  if (warp == 0 && !PAGED) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const int total_units = p.B * p.Hq * p.n_units;
      int item = 0;  // K/V items issued so far (the ring runs on across units)
      int step = 0;  // step ring: steps issued so far
      int slot_rel[STAGES];  // step ring: the step that releases each slot's item (-1: none yet)
#pragma unroll
      for (int i = 0; i < STAGES; ++i) slot_rel[i] = -1;
      int q_uses = 0;
      bool ok = true;
      bool owned = false;       // this CTA's first fetch found or claimed the launch's counter
      bool fetched_last = false;  // this CTA made its final fetch (or needs none)
      for (int n = 0; ok; ++n) {
        // Take the next unit, decode it and publish it (idx -1: no work left).
        const int slot = n % kUnitQ;
        if (!mbar_wait(&unit_empty[slot], ((n / kUnitQ) & 1) ^ 1, 4)) break;
        int idx = static_cast<int>(blockIdx.x);
        if (n > 0) {
          const int c = sched_fetch(p.sched, p.sched_tag, owned, total_units);
          idx = c < 0 ? total_units : static_cast<int>(gridDim.x) + c;
          fetched_last = idx >= total_units;
        }
        Unit<NQ> u;
        if (idx < total_units) {
          u = unit_of<NQ, false>(p, idx);
        } else {
          u.idx = -1;
        }
        unit_q[slot] = u;
        mbar_arrive(&unit_full[slot]);
        if (u.idx < 0) break;
        if (u.T == 0) continue;
        // The previous unit's last S MMA must be done with the Q tiles.
        if (q_uses > 0 && !mbar_wait(q_empty, (q_uses - 1) & 1, 5)) break;
        mbar_expect_tx(q_full, NQ * L::kQBytes);
#pragma unroll
        for (int j = 0; j < NQ; ++j)
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(smem + L::kQOff + j * L::kQBytes + c * (kBM * 128), &tmQ, q_full, c * 64,
                        u.q0 + j * kBM, u.bh);
        ++q_uses;
        if constexpr (kStepRing) {
          // Step t of the unit brings V(t-1) and K(t) (items 2t-1, 2t) on one
          // barrier; a slot is refilled once the step that read it is done.
          for (int t = 0; ok && t <= u.T; ++t, ++step) {
            const int nv = t >= 1 ? 1 : 0, nk = t < u.T ? 1 : 0;
            for (int i = 0; i < nv + nk; ++i) {
              const int r = slot_rel[(item + i) % STAGES];
              if (r >= 0 && !mbar_wait(&step_empty[r % kStepR], (r / kStepR) & 1, 1)) ok = false;
            }
            if (!ok) break;
            uint64_t* bar = &step_full[step % kStepR];
            mbar_expect_tx(bar, (nv + nk) * L::kKVBytes);
            for (int i = 0; i < nv + nk; ++i, ++item) {
              const int st = item % STAGES;
              const bool is_v = i < nv;
              const int tt = is_v ? t - 1 : t;
#pragma unroll
              for (int c = 0; c < L::kDI / 64; ++c)
                tma_load_3d(smem + L::kKVOff + st * L::kKVBytes + c * (kBN * 128), is_v ? &tmV : &tmK, bar,
                            c * 64, (u.tmin + tt) * kBN, u.kvh);
              slot_rel[st] = step;
            }
          }
        } else {
          for (int i = 0; i < 2 * L::kH * u.T; ++i, ++item) {
            const int st = item % STAGES;
            if (!mbar_wait(&kv_empty[st], ((item / STAGES) & 1) ^ 1, 1)) {
              ok = false;
              break;
            }
            mbar_expect_tx(&kv_full[st], L::kKVBytes);
            int t, kind, hh;
            load_item<NQ, L::kH, L::kPSep>(i, u.T, t, kind, hh);
            const CUtensorMap* map = kind ? &tmV : &tmK;
#pragma unroll
            for (int c = 0; c < L::kDI / 64; ++c)
              tma_load_3d(smem + L::kKVOff + st * L::kKVBytes + c * (kBN * 128), map, &kv_full[st],
                          hh * L::kDI + c * 64, (u.tmin + (rev_tiles ? u.T - 1 - t : t)) * kBN, u.kvh);
          }
        }
      }
      // A CTA that stopped early still makes its final fetch, so that the
      // launch's fetches add up and the counter slot is freed.
      while (!fetched_last) {
        const int c = sched_fetch(p.sched, p.sched_tag, owned, total_units);
        fetched_last = c < 0 || static_cast<int>(gridDim.x) + c >= total_units;
      }
      // Drain: never leave the CTA with a copy still writing shared memory
      // (after one wait gives up, the rest are not attempted).
      bool drained = q_uses == 0 || mbar_wait(q_full, (q_uses - 1) & 1, 2);
      if (kStepRing) {
        for (int st = max(0, step - kStepR); drained && st < step; ++st)
          drained = mbar_wait(&step_full[st % kStepR], (st / kStepR) & 1, 3);
      } else {
        for (int it = max(0, item - STAGES); drained && it < item; ++it)
          drained = mbar_wait(&kv_full[it % STAGES], (it / STAGES) & 1, 3);
      }
    }
    __syncwarp();
  } else if (warp == 0 || (PAGED && warp == L::kProd2Warp)) {
    // ---------------------------------------------------------------- TMA producers, paged cache
    // Two whole warps: a key tile spans 128 / page_size pages, each loaded as
    // kDI / 64 boxes; box b of an item goes to lane b / 2 of producer warp
    // b % 2, so each warp issues half of an item's boxes (a warp hands its
    // lanes' copies to the TMA unit one after the other).  Warp 0 takes the
    // units from the work counter and publishes them; the second producer
    // warp reads them from the unit queue.  Lane 0 of each does its waits and
    // its arrival on the item's barrier (two per item); warp 0 loads Q.  Each lane
    // keeps the page id of its box for the tiles t-2 .. t+2 around the latest
    // K(t) (a value tile is loaded at most two key tiles after its own): the
    // block-table read of a tile is issued two tiles ahead of its first use.  Pages past the context's end are not loaded
    // (their keys are masked; their stale rows, real cache rows or zeros, get
    // zero weight).  A value page the context ends inside is loaded on its own
    // barrier; the warp then zeroes its slots past the end before the item is
    // complete, so whatever those cache slots hold never meets a zero weight.
    constexpr uint32_t kFull = 0xFFFFFFFFu;
    constexpr int kNone = -0x7FFFFFFF - 1;  // "no page": past the context or not an issuing lane
    constexpr int kCh = L::kDI / 64;        // boxes per page and item
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
    }
    const int total_units = __ldg(p.unit_prefix + p.num_seqs);
    const int ps = p.page_size;
    const int pw = warp == 0 ? 0 : 1;  // producer warp
    const int b_l = 2 * lane + pw;      // this lane's box of an item
    const int g_l = b_l / kCh;          // its page within a key tile
    const int c_l = b_l % kCh;          // and 64-column box
    const bool issuer = g_l < kBN / ps;
    uint64_t* const tbar = &tail_bar[pw];  // this warp's partly filled value page
    int item = 0, q_uses = 0, tails = 0;
    int step = 0;          // step ring: steps issued so far
    int slot_rel[STAGES];  // step ring: the step that last read each slot (-1: none yet)
#pragma unroll
    for (int i = 0; i < STAGES; ++i) slot_rel[i] = -1;
    bool ok = true;
    bool owned = false;  // lane 0: this CTA's first fetch found or claimed the launch's counter
    // Lane 0: this CTA made its final fetch, or needs none (no first unit;
    // the second producer warp never fetches).
    bool fetched_last = pw == 1 || static_cast<int>(blockIdx.x) >= total_units;
    for (int n = 0; ok; ++n) {
      const int slot = n % kUnitQ;
      Unit<NQ> u;
      if (pw == 0) {
        int idx = -2;
        if (lane == 0 && mbar_wait(&unit_empty[slot], ((n / kUnitQ) & 1) ^ 1, 4)) {
          idx = static_cast<int>(blockIdx.x);
          if (n > 0) {
            const int c = sched_fetch(p.sched, p.sched_tag, owned, total_units);
            idx = c < 0 ? total_units : static_cast<int>(gridDim.x) + c;
            fetched_last = idx >= total_units;
          }
        }
        idx = __shfl_sync(kFull, idx, 0);
        if (idx == -2) break;
        if (idx < total_units) {
          u = unit_of<NQ, true>(p, idx);
        } else {
          u.idx = -1;
        }
        if (lane == 0) {
          unit_q[slot] = u;
          mbar_arrive(&unit_full[slot]);
        }
      } else {
        int got = lane == 0 ? next_unit(n, 27).idx : 0;
        got = __shfl_sync(kFull, got, 0);
        if (got == -2) break;
        __syncwarp();
        u = unit_q[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(&unit_empty[slot]);
      }
      if (u.idx < 0) break;
      if (u.T == 0) continue;
      int qok = 1;
      if (pw == 0 && lane == 0) {
        // The previous unit's last S MMA must be done with the Q tile.
        if (q_uses > 0 && !mbar_wait(q_empty, (q_uses - 1) & 1, 5)) {
          qok = 0;
        } else {
          mbar_expect_tx(q_full, NQ * L::kQBytes);
#pragma unroll
          for (int j = 0; j < NQ; ++j)
#pragma unroll
            for (int c = 0; c < D / 64; ++c)  // packed [total_q][Hq][d]: 128 tokens of one head
              tma_load_3d(smem + L::kQOff + j * L::kQBytes + c * (kBM * 128), &tmQ, q_full, c * 64, u.bh,
                          u.qbase + u.q0 + j * kBM);
        }
      }
      if (!__shfl_sync(kFull, qok, 0)) break;
      if (pw == 0) ++q_uses;
      const long long bt_row = static_cast<long long>(u.seq) * p.max_pages;
      {
        // The block-table entries of the unit's pages into L2 now, one line
        // per lane (16-token pages: a 128-byte line every 4 key tiles), so
        // that their reads two tiles ahead of use never wait on DRAM.
        const long long e0 = bt_row + static_cast<long long>(u.tmin) * kBN / ps;
        const long long e1 = bt_row + (min(static_cast<long long>(u.tmin + u.T) * kBN, static_cast<long long>(u.nk)) + ps - 1) / ps;
        if (e1 > e0) {
          const uintptr_t a = reinterpret_cast<uintptr_t>(p.block_table + e0);
          const uintptr_t b = reinterpret_cast<uintptr_t>(p.block_table + e1 - 1);
          for (uintptr_t line = (a & ~uintptr_t(127)) + uintptr_t(128) * (lane + 32 * pw); line <= b; line += 128 * 64)
            prefetch_line_l2(reinterpret_cast<const void*>(line < a ? a : line));
        }
      }
      auto page_of = [&](int t) -> int {
        const int kp = (u.tmin + t) * kBN + g_l * ps;
        return (issuer && kp < u.nk) ? __ldg(p.block_table + bt_row + kp / ps) : kNone;
      };
      int pg_m2 = kNone, pg_m1 = kNone;
      int pg_cur = page_of(0);
      int pg_next = u.T > 1 ? page_of(1) : kNone;
      int pg_next2 = u.T > 2 ? page_of(2) : kNone;
      int kt_cur = 0;  // tile of the latest K item
      if constexpr (kStepRing) {
        // Step t of the unit brings V(t-1) and K(t) (items 2t-1, 2t) on one
        // barrier: the page boxes of both add their bytes, and the warp
        // arrives once, after zeroing a value tile's slots past the context
        // end.  A slot is refilled once the step that read it is done.
        for (int t = 0; ok && t <= u.T; ++t, ++step) {
          const int nv = t >= 1 ? 1 : 0, nk = t < u.T ? 1 : 0;
          int wok = 1;
          if (lane == 0) {
            for (int i = 0; i < nv + nk; ++i) {
              const int r = slot_rel[(item + i) % STAGES];
              if (r >= 0 && !mbar_wait(&step_empty[r % kStepR], (r / kStepR) & 1, 1)) wok = 0;
            }
          }
          if (!__shfl_sync(kFull, wok, 0)) {
            ok = false;
            break;
          }
          uint64_t* bar = &step_full[step % kStepR];
          for (int i = 0; i < nv + nk; ++i, ++item) {
            const int st = item % STAGES;
            const int kind = i < nv ? 1 : 0;
            const int tt = kind ? t - 1 : t;
            if (kind == 0 && tt > 0) {
              pg_m2 = pg_m1;
              pg_m1 = pg_cur;
              pg_cur = pg_next;
              pg_next = pg_next2;
              pg_next2 = tt + 2 < u.T ? page_of(tt + 2) : kNone;
              kt_cur = tt;
            }
            // V(t-1) comes right before K(t): its pages are tile t-1's.
            const int pg = pg_cur;
            const int kp = (u.tmin + tt) * kBN + g_l * ps;
            const bool valid = pg >= 0 && pg < p.num_pages;
            if (pg != kNone && !valid) report_error(7 /* ATTN_ERR_BOUNDS */, 8, pg);
            const bool is_tail = valid && kind == 1 && kp + ps > u.nk;
            const uint32_t tail_mask = __ballot_sync(kFull, is_tail);
            const uint32_t load_mask = __ballot_sync(kFull, valid && !is_tail);
            if (lane == 0) {
              const uint32_t box = static_cast<uint32_t>(ps) * 128u;
              mbar_expect_tx_only(bar, __popc(load_mask) * box);
              if (tail_mask != 0) mbar_expect_tx(tbar, __popc(tail_mask) * box);
            }
            __syncwarp();
            if (valid)
              tma_load_4d(smem + L::kKVOff + st * L::kKVBytes + c_l * (kBN * 128) + g_l * ps * 128,
                          kind ? &tmV : &tmK, is_tail ? tbar : bar, c_l * 64, u.kvh, 0, pg);
            slot_rel[st] = step;
            if (tail_mask != 0) {
              int tok = 1;
              if (lane == 0) tok = mbar_wait(tbar, tails & 1, 26);
              if (!__shfl_sync(kFull, tok, 0)) {
                ok = false;
                break;
              }
              ++tails;
              // Zero slots [rem, ps) of this warp's box of the tail page (one
              // page holds the context end; a warp has at most one of its boxes).
              const int tb = 2 * (__ffs(tail_mask) - 1) + pw;
              const int tg = tb / kCh, tc = tb % kCh;
              const int rem = u.nk - ((u.tmin + tt) * kBN + tg * ps);
              const int nz = ps - rem;
              const uint32_t stage = sbase + L::kKVOff + st * L::kKVBytes;
              for (int e = lane; e < nz * 8; e += 32) {
                const int k16 = e & 7;
                const int r = rem + (e >> 3);
                st_shared_v4(stage + tc * (kBN * 128) + (tg * ps + r) * 128 + k16 * 16, 0u, 0u, 0u, 0u);
              }
              fence_proxy_async_smem();
              __syncwarp();
            }
          }
          if (!ok) break;
          __syncwarp();
          if (lane == 0) mbar_arrive(bar);  // this warp's one arrival of the step
        }
        continue;
      }
      for (int i = 0; i < 2 * L::kH * u.T; ++i, ++item) {
        const int st = item % STAGES;
        int t, kind, hh;
        load_item<NQ, L::kH, L::kPSep>(i, u.T, t, kind, hh);
        if (kind == 0 && hh == 0 && t > 0) {
          pg_m2 = pg_m1;
          pg_m1 = pg_cur;
          pg_cur = pg_next;
          pg_next = pg_next2;
          pg_next2 = t + 2 < u.T ? page_of(t + 2) : kNone;
          kt_cur = t;
        }
        int wok = 1;
        if (lane == 0) wok = mbar_wait(&kv_empty[st], ((item / STAGES) & 1) ^ 1, 1);
        if (!__shfl_sync(kFull, wok, 0)) {
          ok = false;
          break;
        }
        // K(t) uses tile t's pages; V(t) comes zero to two key tiles later.
        const int back = kind == 0 ? 0 : kt_cur - t;
        const int pg = back == 0 ? pg_cur : (back == 1 ? pg_m1 : pg_m2);
        const int kp = (u.tmin + t) * kBN + g_l * ps;
        const bool valid = pg >= 0 && pg < p.num_pages;
        if (pg != kNone && !valid) report_error(7 /* ATTN_ERR_BOUNDS */, 8, pg);
        const bool is_tail = valid && kind == 1 && kp + ps > u.nk;
        const uint32_t tail_mask = __ballot_sync(kFull, is_tail);
        const uint32_t load_mask = __ballot_sync(kFull, valid && !is_tail);
        if (lane == 0) {
          const uint32_t box = static_cast<uint32_t>(ps) * 128u;
          if (tail_mask == 0) {
            mbar_expect_tx(&kv_full[st], __popc(load_mask) * box);  // arrives; 0 bytes completes at once
          } else {
            mbar_expect_tx_only(&kv_full[st], __popc(load_mask) * box);
            mbar_expect_tx(tbar, __popc(tail_mask) * box);
          }
        }
        __syncwarp();
        const CUtensorMap* map = kind ? &tmV : &tmK;
        if (valid)
          tma_load_4d(smem + L::kKVOff + st * L::kKVBytes + c_l * (kBN * 128) + g_l * ps * 128, map,
                      is_tail ? tbar : &kv_full[st], hh * L::kDI + c_l * 64, u.kvh, 0, pg);
        if (tail_mask != 0) {
          int tok = 1;
          if (lane == 0) tok = mbar_wait(tbar, tails & 1, 26);
          if (!__shfl_sync(kFull, tok, 0)) {
            ok = false;
            break;
          }
          ++tails;
          // Zero slots [rem, ps) of this warp's box of the tail page.
          const int tb = 2 * (__ffs(tail_mask) - 1) + pw;
          const int tg = tb / kCh, tc = tb % kCh;
          const int rem = u.nk - ((u.tmin + t) * kBN + tg * ps);
          const int nz = ps - rem;
          const uint32_t stage = sbase + L::kKVOff + st * L::kKVBytes;
          for (int e = lane; e < nz * 8; e += 32) {
            const int k16 = e & 7;
            const int r = rem + (e >> 3);
            st_shared_v4(stage + tc * (kBN * 128) + (tg * ps + r) * 128 + k16 * 16, 0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&kv_full[st]);  // this warp's one arrival of the item
        }
      }
    }
    if (lane == 0) {
      // A CTA that stopped early still makes its final fetch (see sched_fetch).
      while (!fetched_last) {
        const int c = sched_fetch(p.sched, p.sched_tag, owned, total_units);
        fetched_last = c < 0 || static_cast<int>(gridDim.x) + c >= total_units;
      }
      // Drain: never leave the CTA with a copy still writing shared memory
      // (after one wait gives up, the rest are not attempted).
      bool drained = q_uses == 0 || mbar_wait(q_full, (q_uses - 1) & 1, 2);
      if (kStepRing) {
        for (int st = max(0, step - kStepR); drained && st < step; ++st)
          drained = mbar_wait(&step_full[st % kStepR], (st / kStepR) & 1, 3);
      } else {
        for (int it = max(0, item - STAGES); drained && it < item; ++it)
          drained = mbar_wait(&kv_full[it % STAGES], (it / STAGES) & 1, 3);
      }
    }
    __syncwarp();
  } else if (BIAS == 2 && warp == 2 + 4 * NQ) {
    // ---------------------------------------------------------------- bias loader
    // The bias tile of (query tile, key tile t), in the order the softmax
    // threads consume them; its own ring, so the K/V stream never waits on it.
    if (lane == 0) {
      tma_prefetch_desc(&tmB);
      int bitem = 0;
      bool ok = true;
      for (int n = 0; ok; ++n) {
        const Unit<NQ> u = next_unit(n, 25);
        if (u.idx == -2) break;
        mbar_arrive(&unit_empty[n % kUnitQ]);
        if (u.idx < 0) break;
        const int b = u.bh / p.Hq;
        const int h = u.bh - b * p.Hq;
        for (int i = u.lo[0]; i < u.hi[0]; ++i, ++bitem) {
          const int t = rev_tiles ? u.hi[0] - 1 - (i - u.lo[0]) : i;
          const int bs = bitem % bias_ring<BIAS>();
          if (!mbar_wait(&bias_empty[bs], ((bitem / bias_ring<BIAS>()) & 1) ^ 1, 6)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&bias_full[bs], L::kBiasBytes);
#pragma unroll
          for (int c = 0; c < 2; ++c)
            tma_load_4d(smem + L::kBiasOff + bs * L::kBiasBytes + c * (kBM * 128), &tmB, &bias_full[bs],
                        t * kBN + c * 64, u.q0, h * p.bias_hmul, b * p.bias_bmul);
        }
      }
      for (int it = max(0, bitem - bias_ring<BIAS>()); it < bitem; ++it)
        mbar_wait(&bias_full[it % bias_ring<BIAS>()], (it / bias_ring<BIAS>()) & 1, 7);
    }
    __syncwarp();
  } else if (warp == 1 || (L::kSplit && warp == L::kPVWarp)) {
    // ---------------------------------------------------------------- MMA issuer(s)
    // With separate P slots warp 1 issues the S products and warp kPVWarp the
    // P V products: while one thread waits, the other keeps the tensor pipe
    // fed (an issuing thread blocks until the pipe accepts its MMA).
    const bool pv_thread = warp != 1;
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, kBN, 0, 0);      // Q K-major, K K-major
      constexpr uint32_t kIdescO = idesc_bf16_f32(kBM, L::kDI, 0, 1);   // P K-major (TMEM), V MN-major
      // Descriptor bases, computed once: within a group only compile-time
      // offsets are added (the 14-bit address field cannot carry: every
      // shared-memory address is below 256 KB), so the issuing thread spends
      // its time issuing MMAs rather than building descriptors.
      const uint64_t dq0 = sdesc_sw128(sbase + L::kQOff, 16, 1024);
      const uint64_t dkv0 = sdesc_sw128(sbase + L::kKVOff, 16, 1024);
      const uint64_t dv0 = sdesc_sw128(sbase + L::kKVOff, kBN * 128, 1024);
      int item0 = 0;        // first K/V item of the current unit
      int step = 0;         // step ring: steps consumed so far
      int q_uses = 0;       // units with work so far
      int cnt[2] = {0, 0};  // S tiles issued: per query tile (NQ = 2), in total (NQ = 1, cnt[0])
      int o_uses[2] = {0, 0};
      bool ok = true;

      auto wait_item = [&](int item, int where) {
        return mbar_wait(&kv_full[item % STAGES], (item / STAGES) & 1, where);
      };
      // S = Q_j K_t^T into S slot `slot`; waits for each K item in turn.
      auto issue_s = [&](int j, int slot, int kitem, bool wait) -> bool {
        const uint64_t da = dq0 + static_cast<uint64_t>((j * L::kQBytes) >> 4);
        const uint32_t dst = tmem + L::kSCol + slot * kBN;
#pragma unroll
        for (int hh = 0; hh < L::kH; ++hh) {
          const int item = kitem + hh;
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
      // O_j (+)= P_j V_t: one N = kDI product per V item; `first` overwrites O_j.
      auto issue_pv = [&](int j, int slot, int vitem, bool wait, bool first) -> bool {
        const uint32_t pa = L::kPSep ? tmem + L::kPCol + slot * (kBN / 2) : tmem + L::kSCol + slot * kBN;
#pragma unroll
        for (int hh = 0; hh < L::kH; ++hh) {
          const int item = vitem + hh;
          if (wait) {
            if (!wait_item(item, 11)) return false;
            tc_fence_after();
          }
          const uint64_t db = dv0 + static_cast<uint64_t>(((item % STAGES) * L::kKVBytes) >> 4);
          const uint32_t dst = tmem + j * D + hh * L::kDI;
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            umma_bf16_ts(dst, pa + kk * 8, db + static_cast<uint64_t>((kk * (16 * 128)) >> 4), kIdescO,
                         (!first || kk > 0) ? 1u : 0u);
        }
        return true;
      };
      auto release = [&](int first_item) {
#pragma unroll
        for (int hh = 0; hh < L::kH; ++hh) umma_commit(&kv_empty[(first_item + hh) % STAGES]);
      };
      // Before a unit's first P V into O_j, the previous unit's epilogue must
      // have read O_j out of tensor memory.
      auto wait_o_free = [&](int j) -> bool {
        if (o_uses[j] == 0) return true;
        if (!mbar_wait(&o_free[j], (o_uses[j] - 1) & 1, 16)) return false;
        tc_fence_after();
        return true;
      };

      for (int n = 0; ok; ++n) {
        const Unit<NQ> u = next_unit(n, 17);
        if (u.idx == -2) break;
        mbar_arrive(&unit_empty[n % kUnitQ]);
        if (u.idx < 0) break;
        if (u.T == 0) continue;
        if (!pv_thread) {
          ok = mbar_wait(q_full, q_uses & 1, 10);
          if (!ok) break;
        }
        const int T = u.T;
        if (L::kPSep) {
          // S(c) for the unit's tiles into slot c & 1 as soon as the softmax
          // of tile c - 2 has read that slot, two tiles ahead of the P V
          // products, which read P from its own slots.
          const int c0 = cnt[0];
          auto s_tile = [&](int t) -> bool {
            const int c = c0 + t;
            if (c >= 2) {
              if (!mbar_wait(&s_free[c & 1], ((c - 2) >> 1) & 1, 18)) return false;
              tc_fence_after();
            }
            const int kit = item0 + k_pos<1, true>(t) * L::kH;
            if (!issue_s(0, c & 1, kit, true)) return false;
            umma_commit(&s_full[c & 1]);
            release(kit);
            if (t == T - 1) umma_commit(q_empty);  // the unit's last S MMA is issued
            return true;
          };
          auto pv_tile = [&](int t) -> bool {
            const int c = c0 + t;
            if (!mbar_wait(&p_full[c & 1], (c >> 1) & 1, 12)) return false;
            tc_fence_after();
            if (t == 0 && !wait_o_free(0)) return false;
            const int vit = item0 + v_pos<1, true>(t, T) * L::kH;
            if (!issue_pv(0, c & 1, vit, true, t == 0)) return false;
            umma_commit(&pv_free[c & 1]);
            release(vit);
            if (t == T - 1) {
              umma_commit(&o_done[0]);
              ++o_uses[0];
            }
            return true;
          };
          if (L::kSplit) {
            // This thread's half: every S, or every P V.
            for (int t = 0; ok && t < T; ++t) ok = pv_thread ? pv_tile(t) : s_tile(t);
          } else {
            // One thread: S(0), S(1), then S(t + 2) before P V(t).
            for (int t = 0; ok && t < T && t < 2; ++t) ok = s_tile(t);
            for (int t = 0; ok && t < T; ++t) {
              if (t + 2 < T) {
                ok = s_tile(t + 2);
                if (!ok) break;
              }
              ok = pv_tile(t);
            }
          }
          cnt[0] += T;
        } else {
          for (int t = 0; ok && t <= T; ++t) {
            const int kit = item0 + k_pos<NQ>(t) * L::kH;                      // K(t)
            const int vit = item0 + (t >= 1 ? v_pos<NQ>(t - 1, T) : 0) * L::kH;  // V(t-1)
            const int ta = u.tmin + t;  // absolute key tile of S(t); PV is on tile ta - 1
            if (NQ == 2) {
              // PV_A(t-1), S_A(t), PV_B(t-1), S_B(t); K/V items are waited for
              // by their first user and released after their last.
              bool waitedV = false, waitedK = false;
              if (kStepRing) {
                // Both of the step's items on one barrier (every step reads one).
                ok = mbar_wait(&step_full[step % kStepR], (step / kStepR) & 1, 13);
                if (!ok) break;
                tc_fence_after();
                waitedV = waitedK = true;
              }
#pragma unroll
              for (int j = 0; j < NQ; ++j) {
                if (t >= 1 && ta - 1 >= u.lo[j] && ta - 1 < u.hi[j]) {
                  ok = mbar_wait(&p_full[j], (cnt[j] - 1) & 1, 12);
                  if (!ok) break;
                  tc_fence_after();
                  if (ta - 1 == u.lo[j]) {
                    ok = wait_o_free(j);
                    if (!ok) break;
                  }
                  ok = issue_pv(j, j, vit, !waitedV, ta - 1 == u.lo[j]);
                  if (!ok) break;
                  waitedV = true;
                  if (ta - 1 == u.hi[j] - 1) {
                    umma_commit(&o_done[j]);
                    ++o_uses[j];
                  }
                }
                if (t < T && ta >= u.lo[j] && ta < u.hi[j]) {
                  ok = issue_s(j, j, kit, !waitedK);
                  if (!ok) break;
                  waitedK = true;
                  umma_commit(&s_full[j]);
                  ++cnt[j];
                }
              }
              if (!ok) break;
              if (kStepRing) {
                umma_commit(&step_empty[step % kStepR]);
                ++step;
              } else {
                if (waitedV) release(vit);
                if (waitedK) release(kit);
              }
              if (t == T - 1) umma_commit(q_empty);  // the unit's last S MMA is issued
            } else {
              // S(t) into slot c&1 (overlaps the softmax of tile t-1), then PV(t-1).
              if (t < T) {
                const int c = cnt[0];
                ok = issue_s(0, c & 1, kit, true);
                if (!ok) break;
                umma_commit(&s_full[c & 1]);
                ++cnt[0];
                release(kit);
                if (t == T - 1) umma_commit(q_empty);
              }
              if (t >= 1) {
                const int c = cnt[0] - (t < T ? 2 : 1);  // running index of tile t-1
                ok = mbar_wait(&p_full[c & 1], (c >> 1) & 1, 12);
                if (!ok) break;
                tc_fence_after();
                if (t - 1 == 0) {
                  ok = wait_o_free(0);
                  if (!ok) break;
                }
                ok = issue_pv(0, c & 1, vit, true, t - 1 == 0);
                if (!ok) break;
                umma_commit(pv_done);
                release(vit);
                if (t - 1 == T - 1) {
                  umma_commit(&o_done[0]);
                  ++o_uses[0];
                }
              }
            }
          }
        }
        item0 += 2 * L::kH * T;
        ++q_uses;
      }
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
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t o_cols = lane_base + j * D;
    const float sl = p.scale_log2;
    int cnt = 0;                   // tiles softmaxed so far (running S/P barrier phases)
    int bcnt = 0;                  // staged bias tiles consumed so far
    int o_uses = 0;
    bool ok = true;

    for (int n = 0; ok; ++n) {
      // Lane 0 waits for the entry; after the warp barrier every lane copies it.
      int got = lane == 0 ? next_unit(n, 23).idx : 0;
      got = __shfl_sync(0xFFFFFFFFu, got, 0);
      if (got == -2) break;
      __syncwarp();
      const Unit<NQ> u = unit_q[n % kUnitQ];
      __syncwarp();
      if (lane == 0) mbar_arrive(&unit_empty[n % kUnitQ]);
      if (u.idx < 0) break;
      const int diag = u.nk - u.nq;  // key j allowed for row i iff j <= i + diag (causal)
      const int r0 = u.q0 + j * kBM;
      if (r0 >= u.nq) continue;  // this query tile lies past the problem's rows: nothing to write
      const int qrow = r0 + row;
      const int nt = u.hi[j] > u.lo[j] ? u.hi[j] - u.lo[j] : 0;
      const int bh = u.bh;
      // Biased path (ALiBi slopes and/or a dense bias): scores get an additive
      // term before the max, so the max is taken over the biased, scaled
      // scores.  In base 2: x = s * sl + (alibi * (j - i - diag) + bias) * log2(e).
      constexpr bool biased = BIAS != 0;  // instantiated separately: the plain path keeps its registers
      const int hq = bh % p.Hq;
      const uint16_t* brow = nullptr;
      if (BIAS == 1 && p.bias != nullptr && qrow < u.nq)
        brow = p.bias + static_cast<long long>(bh / p.Hq) * p.bias_sb + static_cast<long long>(hq) * p.bias_sh +
               static_cast<long long>(qrow) * p.Nk;
      // Multiplier of r[] in the exponent: the biased paths keep r[] in
      // natural units (s * scale + alibi * distance + bias) and convert to
      // base 2 there.
      const float mul = biased ? 1.4426950408889634f : sl;
      const float scale_nat = sl * 0.6931471805599453f;
      const float slope = p.alibi != nullptr ? p.alibi[hq] : 0.f;
      // l sums the exact weights (for LSE); lr sums the bf16-rounded weights
      // the P V product uses, so O = o / lr is an exact convex combination of
      // V rows before output rounding.
      float m_ref = -INFINITY;
      float l0 = 0.f, l1 = 0.f, lr0 = 0.f, lr1 = 0.f;

      for (int ti = 0; ti < nt; ++ti) {
        const int t = rev_tiles ? u.hi[j] - 1 - ti : u.lo[j] + ti;  // absolute key tile
        const int slot = NQ == 2 ? j : (cnt & 1);
        const uint32_t s_par = NQ == 2 ? (cnt & 1) : ((cnt >> 1) & 1);
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(&s_full[slot], s_par, 20));
        if (!ok) break;
        tc_fence_after();
        uint32_t r[kBN];
        tmem_ld128(lane_base + L::kSCol + slot * kBN, r);
        if (L::kPSep) {
          // S is in registers: the MMA thread may reuse the slot for S(c + 2).
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&s_free[slot]);
        }

        // Row max of the raw scores (masked keys -> -inf); scale > 0 keeps
        // the order, so the scaled max is mx * sl.  On the biased path r[]
        // first becomes the biased, scaled score and the max is over that.
        const int k0 = t * kBN;
        if (BIAS == 2) {
          // Row `row` of the staged bias tile: 16 chunks of 8 keys, chunk c of
          // a 128-byte row at position c ^ (row & 7) (the TMA 128-byte
          // swizzle), so the 8 rows of each quarter-warp phase hit distinct banks.
          // Per column pair: r = s * scale + (alibi * dist + bias), two paired
          // FMAs; dist = j - i - diag runs in four exact integer-valued chains
          // (one per pair of an 8-key chunk), each advanced by 8 per chunk.
          const float d00 = static_cast<float>(k0 - qrow - diag);
          float dist[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) dist[e] = d00 + static_cast<float>(e);
          const int bs = bcnt % bias_ring<BIAS>();
          ok = __all_sync(0xFFFFFFFFu, mbar_wait(&bias_full[bs], (bcnt / bias_ring<BIAS>()) & 1, 24));
          if (!ok) break;
          const uint32_t brow_s = sbase + L::kBiasOff + bs * L::kBiasBytes + row * 128;
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const uint4 w = ld_shared_v4(brow_s + (c >> 3) * (kBM * 128) + (((c & 7) ^ (row & 7)) << 4));
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int cc = c * 8 + 2 * e;
              float u0, u1, y0, y1;
              ffma2(u0, u1, slope, slope, dist[2 * e], dist[2 * e + 1], bf16lo(ws[e]), bf16hi(ws[e]));
              ffma2(y0, y1, __uint_as_float(r[cc]), __uint_as_float(r[cc + 1]), scale_nat, scale_nat, u0, u1);
              r[cc] = __float_as_uint(y0);
              r[cc + 1] = __float_as_uint(y1);
              fadd2(dist[2 * e], dist[2 * e + 1], dist[2 * e], dist[2 * e + 1], 8.f, 8.f);
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&bias_empty[bs]);
          ++bcnt;
        } else if (biased) {
          // The same terms in the same order as the staged path above.
          const float d00 = static_cast<float>(k0 - qrow - diag);
          if (brow != nullptr) {
            // The row's bias for this tile, read as aligned 32-bit words (the
            // bias buffer is 4-byte aligned; when the tile starts on an odd
            // element the pairs straddle words and are re-paired by a funnel
            // shift).  Words holding no element of this row's tile are not read.
            const uint16_t* a = brow + k0;
            const int odd = static_cast<int>((reinterpret_cast<uintptr_t>(a) >> 1) & 1u);
            const uint32_t* wp = reinterpret_cast<const uint32_t*>(a - odd);
            const int nvalid = u.nk - k0;
            uint32_t wv[kBN / 2 + 1];
#pragma unroll
            for (int i = 0; i <= kBN / 2; ++i) wv[i] = (2 * i - odd < nvalid) ? __ldg(wp + i) : 0u;
#pragma unroll
            for (int i = 0; i < kBN / 2; ++i) {
              const uint32_t pr = __funnelshift_r(wv[i], wv[i + 1], 16u * odd);
              float u0, u1, y0, y1;
              ffma2(u0, u1, slope, slope, d00 + static_cast<float>(2 * i), d00 + static_cast<float>(2 * i + 1),
                    bf16lo(pr), bf16hi(pr));
              ffma2(y0, y1, __uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]), scale_nat, scale_nat, u0, u1);
              r[2 * i] = __float_as_uint(y0);
              r[2 * i + 1] = __float_as_uint(y1);
            }
          } else {
#pragma unroll
            for (int cc = 0; cc < kBN; cc += 2) {
              float u0, u1, y0, y1;
              ffma2(u0, u1, slope, slope, d00 + static_cast<float>(cc), d00 + static_cast<float>(cc + 1), 0.f, 0.f);
              ffma2(y0, y1, __uint_as_float(r[cc]), __uint_as_float(r[cc + 1]), scale_nat, scale_nat, u0, u1);
              r[cc] = __float_as_uint(y0);
              r[cc + 1] = __float_as_uint(y1);
            }
          }
        }
        const bool need_mask = (k0 + kBN > u.nk) || (p.causal && (k0 + kBN - 1 > r0 + diag)) ||
                               (p.window > 0 && k0 <= r0 + kBM - 1 + diag - p.window);
        if (need_mask) {
          const int hi_c = (p.causal ? min(u.nk - 1, qrow + diag) : u.nk - 1) - k0;
          const int lo_c = p.window > 0 ? qrow + diag - p.window + 1 - k0 : -1;
#pragma unroll
          for (int cc = 0; cc < kBN; ++cc)
            if (cc > hi_c || cc < lo_c) r[cc] = 0xFF800000u;  // -inf
        }
        float mx[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) mx[i] = -INFINITY;
#pragma unroll
        for (int cc = 0; cc < kBN; cc += 8) {
          const int a = (cc >> 3) & 3;
          mx[a] = fmax3(mx[a], __uint_as_float(r[cc]), __uint_as_float(r[cc + 1]));
          mx[a] = fmax3(mx[a], __uint_as_float(r[cc + 2]), __uint_as_float(r[cc + 3]));
          mx[a] = fmax3(mx[a], __uint_as_float(r[cc + 4]), __uint_as_float(r[cc + 5]));
          mx[a] = fmax3(mx[a], __uint_as_float(r[cc + 6]), __uint_as_float(r[cc + 7]));
        }
        const float mt = fmaxf(fmax3(mx[0], mx[1], mx[2]), mx[3]) * mul;
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
        for (int cc = 0; cc < kBN; cc += 2) {
          float a0, a1;
          ffma2(a0, a1, __uint_as_float(r[cc]), __uint_as_float(r[cc + 1]), mul, mul, neg_m, neg_m);
          const float p0 = ex2(a0);
          const float p1 = ex2(a1);
          fadd2(l0, l1, l0, l1, p0, p1);
          const uint32_t w = pack_bf16(p0, p1);
          add_bf16x2(lr0, lr1, w);
          pk[cc >> 1] = w;
        }

        if (ti > 0 && __any_sync(0xFFFFFFFFu, rescale)) {
          if (NQ == 1) {
            // O holds tile t-1's contribution only once PV(t-1) is complete;
            // P V products are counted like the tiles (one per tile).
            ok = __all_sync(0xFFFFFFFFu,
                            L::kPSep ? mbar_wait(&pv_free[(cnt - 1) & 1], ((cnt - 1) >> 1) & 1, 21)
                                     : mbar_wait(pv_done, (cnt - 1) & 1, 21));
            if (!ok) break;
            tc_fence_after();
          }
#pragma unroll 1
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32(o_cols + cc * 32, o);
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              float y0, y1;
              ffma2(y0, y1, __uint_as_float(o[i]), __uint_as_float(o[i + 1]), alpha, alpha, 0.f, 0.f);
              o[i] = __float_as_uint(y0);
              o[i + 1] = __float_as_uint(y1);
            }
            tmem_st32(o_cols + cc * 32, o);
          }
        }
        // P over the first half of the S slot, then hand it to the MMA thread.
        if (L::kPSep) {
          // P slot `slot` is free once the P V product of tile cnt - 2 is done.
          if (cnt >= 2) {
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(&pv_free[slot], ((cnt - 2) >> 1) & 1, 27));
            if (!ok) break;
            tc_fence_after();
          }
          tmem_st64(lane_base + L::kPCol + slot * (kBN / 2), pk);
        } else {
          tmem_st64(lane_base + L::kSCol + slot * kBN, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[slot]);
        ++cnt;
      }
      if (!ok) break;

      if (nt > 0) {
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(&o_done[j], o_uses & 1, 22));
        if (!ok) break;
        tc_fence_after();
      }
      // Every lane runs the (warp-collective) TMEM loads; only rows < Nq store.
      const bool store = qrow < u.nq;
      const float lr = lr0 + lr1;
      const float l = l0 + l1;
      const float inv = (lr > 0.f) ? 1.f / lr : 0.f;
      // Plain: O [B*Hq][Nq][d], LSE [B*Hq][Nq].  Paged: O [total_q][Hq][d], LSE [total_q][Hq].
      const size_t lse_off = PAGED ? static_cast<size_t>(u.qbase + qrow) * p.Hq + bh
                                   : static_cast<size_t>(bh) * p.Nq + qrow;
      const size_t row_off = lse_off * D;
      // bf16 rows start 32-byte aligned when O does (a row is 128 bytes or more).
      const bool o32 = (reinterpret_cast<uintptr_t>(p.o) & 31u) == 0;
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        if (nt > 0) {
          tmem_ld32(o_cols + cc * 32, o);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0u;
        }
        if (nt > 0 && cc == D / 32 - 1) {
          // O_j has been read: the next unit's first P V may overwrite it.
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&o_free[j]);
        }
        if (!store) continue;
        if (p.o_f32) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + row_off + cc * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(__uint_as_float(o[4 * i]) * inv, __uint_as_float(o[4 * i + 1]) * inv,
                                 __uint_as_float(o[4 * i + 2]) * inv, __uint_as_float(o[4 * i + 3]) * inv);
        } else if (o32) {
          // Full 32-byte sectors per store (the row's 64 bytes of this chunk).
          uint16_t* dst = static_cast<uint16_t*>(p.o) + row_off + cc * 32;
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int e = 16 * i;
            uint32_t w[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
              w[k] = pack_bf16(__uint_as_float(o[e + 2 * k]) * inv, __uint_as_float(o[e + 2 * k + 1]) * inv);
            st_global_v8(dst + 16 * i, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
          }
        } else {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + row_off + cc * 32);
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
      if (nt > 0) ++o_uses;
      if (store)
        p.lse[lse_off] =
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


// Dispatch order and unit prefix sums of a paged chunked prefill (one block).
// Sequences are handed out longest context first (ties by index), so the
// persistent grid ends on short units rather than on one long sequence; up to
// 1024 sequences are ranked (one per thread), more keep their given order.
// Sequence s gets ceil(q_len / unit_rows) * Hq units (unit_rows = 128 x query
// tiles per unit).  A sequence whose lengths are inconsistent (negative, past
// total_q, or a context longer than its block-table row) is flagged in the
// status word and gets no units, so nothing of it is read.
__global__ void __launch_bounds__(1024) paged_plan_kernel(const int32_t* cu_q, const int32_t* seqlens_k,
                                                         int num_seqs, int total_q, int Hq, int max_pages,
                                                         int page_size, int unit_rows, int32_t* unit_prefix,
                                                         int32_t* seq_order) {
  __shared__ int part[1024];
  __shared__ int key[1024];
  __shared__ int order[1024];
  const int tid = static_cast<int>(threadIdx.x);
  const bool ranked = num_seqs <= 1024;
  auto units = [&](int s, bool report) -> int {
    const int a = cu_q[s], b = cu_q[s + 1], k = seqlens_k[s];
    const bool bad = a < 0 || b < a || b > total_q || k < 0 ||
                     static_cast<long long>(k) > static_cast<long long>(max_pages) * page_size;
    if (bad) {
      if (report) report_error(7 /* ATTN_ERR_BOUNDS */, 9, s);
      return 0;
    }
    return ((b - a + unit_rows - 1) / unit_rows) * Hq;
  };
  if (ranked) {
    if (tid < num_seqs) key[tid] = seqlens_k[tid];
    __syncthreads();
    if (tid < num_seqs) {
      const int k = key[tid];
      int rank = 0;
      for (int j = 0; j < num_seqs; ++j) rank += (key[j] > k || (key[j] == k && j < tid)) ? 1 : 0;
      order[rank] = tid;
    }
    __syncthreads();
  }
  auto seq_at = [&](int r) { return ranked ? order[r] : r; };
  const int per = (num_seqs + blockDim.x - 1) / blockDim.x;
  const int r0 = min(num_seqs, tid * per);
  const int r1 = min(num_seqs, r0 + per);
  int sum = 0;
  for (int r = r0; r < r1; ++r) sum += units(seq_at(r), true);
  part[tid] = sum;
  __syncthreads();
  // Exclusive scan of the per-thread sums (Hillis-Steele over 1024 entries).
  for (int off = 1; off < 1024; off <<= 1) {
    const int v = tid >= off ? part[tid - off] : 0;
    __syncthreads();
    part[tid] += v;
    __syncthreads();
  }
  int run = tid > 0 ? part[tid - 1] : 0;
  for (int r = r0; r < r1; ++r) {
    const int s = seq_at(r);
    unit_prefix[r] = run;
    seq_order[r] = s;
    run += units(s, false);
  }
  if (tid == blockDim.x - 1) unit_prefix[num_seqs] = part[blockDim.x - 1];
}

}  // namespace attn
