// C entry points of the attention backward (declared in include/attn.h);
// included at the end of attn_api.cu so that it shares that translation
// unit's device status word, launch counter and tensor-map helpers.
#pragma once

#include "bwd.cuh"
#include "bwd_wide.cuh"

namespace {

size_t bwd_align(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }

// 3-D f32 map over the dQ accumulator [B*Hq][Nq][d]; one box is [128 rows][32
// columns], 128-byte swizzled (the staging layout of the backward kernel).
bool encode_dq_map(CUtensorMap* map, void* base, int d, int rows, int heads) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4, static_cast<cuuint64_t>(rows) * d * 4};
  cuuint32_t box[3] = {32, 128, 1};
  return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int D, int STAGES, bool BIAS>
attn_status launch_bwd(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mdo,
                       const CUtensorMap& mdq, const attn::BwdParams& p, cudaStream_t stream) {
  using L = attn::BwdLayout<D, STAGES>;
  auto kern = attn::attn_bwd_kernel<D, STAGES, BIAS>;
  if (!ensure_smem<attn::attn_bwd_kernel<D, STAGES, BIAS>>(L::kAlloc)) return ATTN_ERR_LAUNCH;
  const long long grid = static_cast<long long>(p.B) * p.Hkv * ((p.Nk + 127) / 128);
  if (grid > 0x7FFFFFFFLL) return ATTN_ERR_UNSUPPORTED;
  if (grid == 0) return ATTN_OK;
  kern<<<dim3(static_cast<unsigned>(grid)), L::kThreads, L::kAlloc, stream>>>(mq, mk, mv, mdo, mdq, p);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return ATTN_OK;
}

// Head dims served by the 64-query-item kernel (bwd_wide.cuh).  Its dQ
// chunks are [32 queries][128 head-dim columns] f32, unswizzled, added into
// the f32 accumulator [B*Hq][Nq][d].
bool bwd_uses_wide(int d) { return d >= 128; }

bool encode_dq_rows_map(CUtensorMap* map, void* base, int d, int rows, int heads) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(heads)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4, static_cast<cuuint64_t>(rows) * d * 4};
  cuuint32_t box[3] = {128, 32, 1};
  return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

template <int D, int STAGES, bool BIAS>
attn_status launch_bwd_wide(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                            const CUtensorMap& mdo, const CUtensorMap& mdq, const CUtensorMap& mdk,
                            const CUtensorMap& mdv, const attn::BwdParams& p, cudaStream_t stream) {
  using L = attn::BwdWideLayout<D, STAGES>;
  if (!ensure_smem<attn::attn_bwd_wide_kernel<D, STAGES, BIAS>>(L::kAlloc)) return ATTN_ERR_LAUNCH;
  // kSplit CTAs (head-dim halves) per (key tile, batch, kv head), key tile 0 first.
  const long long grid = static_cast<long long>(L::kSplit) * p.B * p.Hkv * ((p.Nk + 127) / 128);
  if (grid > 0x7FFFFFFFLL) return ATTN_ERR_UNSUPPORTED;
  if (grid == 0) return ATTN_OK;
  attn::attn_bwd_wide_kernel<D, STAGES, BIAS>
      <<<dim3(static_cast<unsigned>(grid)), L::kThreads, L::kAlloc, stream>>>(mq, mk, mv, mdo, mdq, mdk, mdv, p);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return ATTN_OK;
}

// Bytes of the f32 dQ accumulator for head dim d.
size_t bwd_acc_bytes(int B, int Hq, int Nq, int d) {
  return static_cast<size_t>(B) * Hq * static_cast<size_t>(Nq) * d * sizeof(float);
}

bool bwd_head_dim_ok(int d) { return d == 64 || d == 128 || d == 256; }

template <bool BIAS>
attn_status launch_bwd_d(int d, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                         const CUtensorMap& mdo, const CUtensorMap& mdq, const CUtensorMap& mdk,
                         const CUtensorMap& mdv, const attn::BwdParams& p, cudaStream_t s) {
  return d == 64    ? launch_bwd<64, 3, BIAS>(mq, mk, mv, mdo, mdq, p, s)
         : d == 128 ? launch_bwd_wide<128, 3, BIAS>(mq, mk, mv, mdo, mdq, mdk, mdv, p, s)
                    : launch_bwd_wide<256, 1, BIAS>(mq, mk, mv, mdo, mdq, mdk, mdv, p, s);
}

attn_status bwd_impl(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                     void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal,
                     float scale, const attn_mask* mask, attn_dtype grad_dtype, void* workspace,
                     size_t workspace_bytes, attn_stream_t stream);

}  // namespace

extern "C" {

size_t attn_bwd_workspace_size(int B, int Hq, int Nq, int d) {
  if (B < 0 || Hq <= 0 || Nq < 0 || !bwd_head_dim_ok(d)) return 0;
  const size_t rows = static_cast<size_t>(B) * Hq * Nq;
  return bwd_align(rows * sizeof(float)) + bwd_align(bwd_acc_bytes(B, Hq, Nq, d));
}

attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                     void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal,
                     float scale, attn_dtype grad_dtype, void* workspace, size_t workspace_bytes,
                     attn_stream_t stream) {
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, Nq, Nk, d, causal, scale, nullptr, grad_dtype,
                  workspace, workspace_bytes, stream);
}

attn_status attn_bwd_masked(const void* q, const void* k, const void* v, const void* o, const void* dout,
                            const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nk,
                            int d, int causal, float scale, const attn_mask* mask, attn_dtype grad_dtype,
                            void* workspace, size_t workspace_bytes, attn_stream_t stream) {
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, Nq, Nk, d, causal, scale, mask, grad_dtype,
                  workspace, workspace_bytes, stream);
}

}  // extern "C"

namespace {

attn_status bwd_impl(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                     void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal,
                     float scale, const attn_mask* mask, attn_dtype grad_dtype, void* workspace,
                     size_t workspace_bytes, attn_stream_t stream) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Nq < 0 || Nk < 0) return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (grad_dtype != ATTN_BF16 && grad_dtype != ATTN_F32) return ATTN_ERR_INVALID_ARG;
  if (!bwd_head_dim_ok(d)) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * Hq > 0x7FFFFFFFLL) return ATTN_ERR_UNSUPPORTED;
  const bool biased = mask != nullptr && (mask->window_left != 0 || mask->alibi_slopes || mask->bias);
  if (biased) {
    if (mask->window_left < 0 || mask->bias_stride_b < 0 || mask->bias_stride_h < 0) return ATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(mask->alibi_slopes) & 3u) || (reinterpret_cast<uintptr_t>(mask->bias) & 3u))
      return ATTN_ERR_MISALIGNED;
  }
  if (B == 0 || (Nq == 0 && Nk == 0)) return ATTN_OK;
  if (Nq > 0 && (!aligned16(q) || !aligned16(o) || !aligned16(dout) || !aligned16(lse) || !aligned16(dq)))
    return ATTN_ERR_MISALIGNED;
  if (Nk > 0 && (!aligned16(k) || !aligned16(v) || !aligned16(dk) || !aligned16(dv))) return ATTN_ERR_MISALIGNED;
  const size_t need = attn_bwd_workspace_size(B, Hq, Nq, d);
  if (!aligned16(workspace) || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
  attn_status st = check_device();
  if (st != ATTN_OK) return st;

  const size_t rows = static_cast<size_t>(B) * Hq * Nq;
  float* dsum = static_cast<float*>(workspace);
  // f32 gradients: dQ is accumulated in place in the caller's dq (zeroed by
  // the prep kernel), so no conversion pass follows; bf16: in the workspace.
  const bool dq_in_place = grad_dtype == ATTN_F32;
  float* dq_acc = dq_in_place ? static_cast<float*>(dq)
                              : reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                                         bwd_align(rows * sizeof(float)));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int sms = sm_count();
  if (rows > 0) {
    const long long blocks = std::min<long long>((static_cast<long long>(rows) * d / 8 + 255) / 256, 16LL * sms);
    attn::bwd_prep_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dout), dsum, dq_acc,
        static_cast<long long>(rows), d, static_cast<long long>(bwd_acc_bytes(B, Hq, Nq, d) / 16));
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
    g_launches.fetch_add(1, std::memory_order_relaxed);
  }

  if (Nk > 0) {
    CUtensorMap mq, mk, mv, mdo, mdq;
    // With Nq == 0 no query tile is ever loaded; the Q / dO maps then describe k.
    const void* qb = Nq > 0 ? q : k;
    const void* db = Nq > 0 ? dout : k;
    const int nq_map = Nq > 0 ? Nq : Nk;
    const int bh_map = Nq > 0 ? B * Hq : B * Hkv;
    const int qbox = bwd_uses_wide(d) ? 64 : 128;
    if (!encode_rows_map(&mq, qb, d, nq_map, bh_map, qbox) || !encode_rows_map(&mdo, db, d, nq_map, bh_map, qbox) ||
        !encode_rows_map(&mk, k, d, Nk, B * Hkv, 128) || !encode_rows_map(&mv, v, d, Nk, B * Hkv, 128))
      return ATTN_ERR_LAUNCH;
    // With Nq == 0 no dQ chunk is ever written; the map then describes one row.
    void* acc_base = Nq > 0 ? static_cast<void*>(dq_acc) : workspace;
    const bool acc_ok = bwd_uses_wide(d) ? encode_dq_rows_map(&mdq, acc_base, d, Nq > 0 ? Nq : 1, Nq > 0 ? B * Hq : 1)
                                         : encode_dq_map(&mdq, acc_base, d, Nq > 0 ? Nq : 1, Nq > 0 ? B * Hq : 1);
    if (!acc_ok) return ATTN_ERR_LAUNCH;
    // bf16 dK, dV leave the 64-query kernel by TMA stores ([128 keys][64
    // columns] boxes, like the K and V loads); f32 ones by direct stores (the
    // maps then describe k and are not used).
    CUtensorMap mdk, mdv;
    const bool bf16_out = grad_dtype == ATTN_BF16;
    if (!encode_rows_map(&mdk, bf16_out ? dk : k, d, Nk, B * Hkv, 128) ||
        !encode_rows_map(&mdv, bf16_out ? dv : k, d, Nk, B * Hkv, 128))
      return ATTN_ERR_LAUNCH;
    attn::BwdParams p;
    p.dk = dk;
    p.dv = dv;
    p.dq_acc = dq_acc;
    p.lse = lse;
    p.dsum = dsum;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.Nq = Nq;
    p.Nk = Nk;
    p.causal = causal ? 1 : 0;
    p.g_f32 = grad_dtype == ATTN_F32 ? 1 : 0;
    p.scale = scale;
    p.scale_log2 = scale * 1.4426950408889634f;
    // Head groups for the 64-query kernel's block order: as many (batch, kv
    // head) pairs as keep their Q, dO and f32 dQ accumulator (8 bytes per
    // query element) within ~64 MB of L2.
    {
      const long long per_pair = static_cast<long long>(Hq / Hkv) * Nq * d * 8;
      long long g = per_pair > 0 ? (64LL << 20) / per_pair : static_cast<long long>(B) * Hkv;
      g = std::max(1LL, std::min(g, static_cast<long long>(B) * Hkv));
      p.head_group = static_cast<int>(g);
    }
    p.window_left = biased ? mask->window_left : 0;
    p.alibi = biased ? mask->alibi_slopes : nullptr;
    p.bias = biased ? static_cast<const uint16_t*>(mask->bias) : nullptr;
    p.bias_sb = biased ? mask->bias_stride_b : 0;
    p.bias_sh = biased ? mask->bias_stride_h : 0;
    // A left window alone needs no bias term: every variant applies it.
    const bool bias_terms = p.alibi != nullptr || p.bias != nullptr;
    st = bias_terms ? launch_bwd_d<true>(d, mq, mk, mv, mdo, mdq, mdk, mdv, p, s)
                : launch_bwd_d<false>(d, mq, mk, mv, mdo, mdq, mdk, mdv, p, s);
    if (st != ATTN_OK) return st;
  }

  if (rows > 0 && !dq_in_place) {
    const long long n4 = static_cast<long long>(rows) * d / 4;
    const long long blocks = std::min<long long>((n4 + 255) / 256, 8LL * sms);
    attn::bwd_post_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(dq_acc, dq, n4, 0);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
    g_launches.fetch_add(1, std::memory_order_relaxed);
  }
  return ATTN_OK;
}

}  // namespace
