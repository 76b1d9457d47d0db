// Prefill attention on sm_103a: TMA-fed shared-memory K/V ring, tcgen05 MMAs
// accumulating S = Q K^T and O += P V in tensor memory, online softmax in
// registers.
//
// Method ("FlashAttention" learn page, aiunderstanding.org, "Technical
// insight"; FAQ on computing softmax without seeing every score): tiles of
// Q, K and V are brought on chip, a running row maximum m and row sum l are
// kept, and the partial output is rescaled whenever m grows, so the final
// normalisation is exact and the N x N score matrix never leaves the SM.
// Key tiles that a row block cannot see (causal future, outside the local
// window of the Arabic context-length thread, point 1) are skipped.
//
// CTA layout (384 threads, one CTA per SM):
//   warp 0      TMA producer: Q tiles once, then K_j, V_j into a STAGES-deep ring
//   warp 1      MMA issuer (lane 0): S_i = Q_i K_j^T, O_i += P_i V_j
//   warp 2      tensor-memory allocator
//   warp 3      idle
//   warps 4-7   softmax + epilogue for Q tile 0 (rows  0..127 of the block)
//   warps 8-11  softmax + epilogue for Q tile 1 (rows 128..255 of the block)
// The MMA order PV_0(j), S_0(j+1), PV_1(j), S_1(j+1) lets one Q tile's
// softmax run while the tensor core works on the other tile.
//
// Tensor memory (512 columns x 128 lanes of 32 bit):
//   S_0 cols [0,128)   S_1 cols [128,256)   O_0 [256,256+D)   O_1 [256+D,256+2D)
//   P_i (bf16 pairs) overwrites cols [0,64) of S_i once S_i is in registers.
#pragma once

#include "ptx.cuh"

namespace b300 {

__device__ unsigned int g_prefill_status;  // OR of kStatus* bits (bounded waits that ran out)

constexpr unsigned kStatusProducer = 1u, kStatusMma = 2u, kStatusSoftmax = 4u;

struct PrefillParams {
  void* o;
  float* lse;
  int B, Hq, Hkv, N;
  int causal, window, o_f32;
  int nqb;           // number of 256-row query blocks
  float scale_log2;  // scale * log2(e): scores are kept in base-2 units
};

template <int D>
struct PrefillCfg {
  static constexpr int BM = 128;  // query rows per Q tile (one softmax warpgroup)
  static constexpr int BN = 128;  // keys per K/V tile
  static constexpr int DCH = D / 64;  // 128-byte swizzle atoms across d
  static constexpr int TILE_BYTES = BM * D * 2;  // one Q, K or V tile (bf16)
  static constexpr int STAGES = (D == 128) ? 4 : 8;
  static constexpr int RING_OFF = 2 * TILE_BYTES;
  static constexpr int BAR_OFF = RING_OFF + STAGES * TILE_BYTES;
  static constexpr int SMEM_BYTES = BAR_OFF + 512 + 1024;  // + barriers + alignment slack
  static constexpr int THREADS = 384;
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(BM == BN, "Q and K/V tiles share one byte layout");
};


template <int D>
__global__ void __launch_bounds__(384, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
  using C = PrefillCfg<D>;
  constexpr int BN = C::BN;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sRing = smem + C::RING_OFF;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = kv_full + STAGES;
  uint64_t* s_full = kv_empty + STAGES;  // [2]
  uint64_t* p_full = s_full + 2;         // [2]
  uint64_t* o_full = p_full + 2;         // [2]
  uint64_t* mma_done = o_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- which (query block, head, batch) this CTA owns; causal: heaviest first
  const int BH = p.B * p.Hq;
  int qb = blockIdx.x / BH;
  if (p.causal) qb = p.nqb - 1 - qb;
  const int bh = blockIdx.x % BH;
  const int b = bh / p.Hq;
  const int h = bh % p.Hq;
  const int hk = h / (p.Hq / p.Hkv);
  const int N = p.N;

  // ---- key-tile range [jlo, jhi] of each Q tile
  int jlo[2], jhi[2];
  bool act[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r0 = qb * 256 + i * 128;
    act[i] = r0 < N;
    const int r1 = min(r0 + 127, N - 1);
    const int klo = (p.window >= 0) ? max(0, r0 - p.window) : 0;
    const int khi = p.causal ? r1 : ((p.window >= 0) ? min(N - 1, r1 + p.window) : N - 1);
    jlo[i] = klo / BN;
    jhi[i] = khi / BN;
  }
  const int J0 = act[1] ? min(jlo[0], jlo[1]) : jlo[0];
  const int J1 = act[1] ? max(jhi[0], jhi[1]) : jhi[0];

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
      mbar_init(&o_full[i], 1);
    }
    mbar_init(mma_done, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ================================================================ producer
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, 2 * C::TILE_BYTES);
      for (int i = 0; i < 2; ++i)
        for (int c = 0; c < C::DCH; ++c)
          tma_load_4d(sQ + i * C::TILE_BYTES + c * (C::BM * 128), &tm_q, q_full, c * 64, h,
                      qb * 256 + i * 128, b);
      const int nloads = 2 * (J1 - J0 + 1);  // K_j, V_j alternate in the ring
      int issued = 0;
      for (; issued < nloads; ++issued) {
        const int s = issued % STAGES;
        if (issued >= STAGES &&
            !mbar_wait(&kv_empty[s], ((issued / STAGES) - 1) & 1, &g_prefill_status,
                       kStatusProducer))
          break;
        mbar_arrive_expect_tx(&kv_full[s], C::TILE_BYTES);
        const int j = J0 + issued / 2;
        const CUtensorMap* tm = (issued & 1) ? &tm_v : &tm_k;
        for (int c = 0; c < C::DCH; ++c)
          tma_load_4d(sRing + s * C::TILE_BYTES + c * (BN * 128), tm, &kv_full[s], c * 64, hk,
                      j * BN, b);
      }
      // Every issued copy has landed before the CTA may exit (a no-op wait on
      // the normal path, where the MMA warp already consumed them all).
      for (int u = max(0, issued - STAGES); u < issued; ++u)
        mbar_wait(&kv_full[u % STAGES], (u / STAGES) & 1, &g_prefill_status, kStatusProducer);
      mbar_wait(q_full, 0, &g_prefill_status, kStatusProducer);
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      const uint32_t idS = idesc_bf16_f32(128, BN, false);
      const uint32_t idO = idesc_bf16_f32(128, D, true);
      const uint32_t sq = smem_u32(sQ);
      const uint32_t sr = smem_u32(sRing);
      uint32_t pcnt[2] = {0u, 0u};

      // S_i = Q_i K^T: K-major operands, 16 elements of d per instruction.
      auto issue_S = [&](int i, int stage) {
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * (C::BM * 128) + (k & 3) * 32;
          const uint64_t a = smem_desc_sw128(sq + i * C::TILE_BYTES + off, 16, 1024);
          const uint64_t bd = smem_desc_sw128(sr + stage * C::TILE_BYTES + off, 16, 1024);
          umma_ss(tmem + i * 128, a, bd, idS, k > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[i]);
      };
      // O_i += P_i V: P (bf16 pairs) from tensor memory, V MN-major in shared
      // memory, 16 keys per instruction.
      auto issue_PV = [&](int i, int stage, bool accumulate) {
#pragma unroll
        for (int k = 0; k < BN / 16; ++k) {
          const uint64_t bd = smem_desc_sw128(sr + stage * C::TILE_BYTES + k * 16 * 128,
                                              BN * 128, 1024);
          umma_ts(tmem + 256 + i * D, tmem + i * 128 + k * 8, bd, idO,
                  (accumulate || k > 0) ? 1u : 0u);
        }
      };

      bool ok = mbar_wait(q_full, 0, &g_prefill_status, kStatusMma);
      if (ok) ok = mbar_wait(&kv_full[0], 0, &g_prefill_status, kStatusMma);
      if (ok) {
        tc_fence_after();
        for (int i = 0; i < 2; ++i)
          if (act[i] && J0 >= jlo[i] && J0 <= jhi[i]) issue_S(i, 0);
        umma_commit(&kv_empty[0]);
      }
      int t = 1;  // ring position of V_j
      for (int j = J0; j <= J1 && ok; ++j, t += 2) {
        const int sv = t % STAGES;
        if (!(ok = mbar_wait(&kv_full[sv], (t / STAGES) & 1, &g_prefill_status, kStatusMma)))
          break;
        tc_fence_after();
        const bool has_next = j < J1;
        const int sk = (t + 1) % STAGES;
        bool k_ready = false;
        for (int i = 0; i < 2 && ok; ++i) {
          if (act[i] && j >= jlo[i] && j <= jhi[i]) {
            if (!(ok = mbar_wait(&p_full[i], pcnt[i] & 1, &g_prefill_status, kStatusMma))) break;
            ++pcnt[i];
            tc_fence_after();
            issue_PV(i, sv, j != jlo[i]);
            if (j == jhi[i]) umma_commit(&o_full[i]);
          }
          if (has_next && act[i] && j + 1 >= jlo[i] && j + 1 <= jhi[i]) {
            if (!k_ready) {
              if (!(ok = mbar_wait(&kv_full[sk], ((t + 1) / STAGES) & 1, &g_prefill_status,
                                   kStatusMma)))
                break;
              tc_fence_after();
              k_ready = true;
            }
            issue_S(i, sk);
          }
        }
        if (!ok) break;
        umma_commit(&kv_empty[sv]);
        if (has_next) {
          if (!k_ready &&
              !(ok = mbar_wait(&kv_full[sk], ((t + 1) / STAGES) & 1, &g_prefill_status,
                               kStatusMma)))
            break;
          umma_commit(&kv_empty[sk]);
        }
      }
      // All MMAs of this CTA complete before tensor memory is released.
      umma_commit(mma_done);
      mbar_wait(mma_done, 0, &g_prefill_status, kStatusMma);
    }
  } else if (warp >= 4) {
    // ================================================================ softmax
    const int i = (warp - 4) >> 2;   // Q tile of this warpgroup
    const int quarter = warp & 3;    // tensor-memory lane quarter this warp may access
    const int r = quarter * 32 + lane;
    const int r0 = qb * 256 + i * 128;
    const int row = r0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_off + i * 128;
    const uint32_t tO = tmem + lane_off + 256 + i * D;
    const float sl2 = p.scale_log2;
    const bool causal = p.causal != 0;
    const int window = p.window;
    float m_ref = -INFINITY;  // base-2 running maximum actually used for P
    float l = 0.f;
    bool ok = true;
    if (act[i]) {
      int n = 0;
      for (int j = jlo[i]; j <= jhi[i]; ++j, ++n) {
        ok = mbar_wait(&s_full[i], n & 1, &g_prefill_status, kStatusSoftmax);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        float s[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t u[32];
          tmem_ld32_wait(tS + c * 32, u);
#pragma unroll
          for (int e = 0; e < 32; ++e) s[c * 32 + e] = __uint_as_float(u[e]);
        }
        const int kv0 = j * BN;
        const bool need_mask =
            (kv0 + BN > N) || (causal && kv0 + BN - 1 > r0) ||
            (window >= 0 && (r0 + 127 - kv0 > window || (!causal && kv0 + BN - 1 - r0 > window)));
        if (need_mask) {
#pragma unroll
          for (int c = 0; c < 128; ++c) {
            const int key = kv0 + c;
            bool vis = key < N;
            if (causal) vis = vis && key <= row;
            if (window >= 0) vis = vis && (row - key <= window) && (causal || key - row <= window);
            if (!vis) s[c] = -INFINITY;
          }
        }
        float mx = s[0];
#pragma unroll
        for (int c = 1; c < 128; ++c) mx = fmaxf(mx, s[c]);
        const float m_new = fmaxf(m_ref, mx * sl2);
        const bool resc = m_new > m_ref + kRescaleThreshold;
        float alpha = 1.f;
        if (resc) {
          alpha = ex2_approx(m_ref - m_new);  // 0 when m_ref = -inf
          m_ref = m_new;
          l *= alpha;
        }
        const float neg_mu = (m_ref == -INFINITY) ? 0.f : -m_ref;
        // P = 2^(s*scale*log2e - m), row sum in f32, bf16 pairs into tensor memory
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float p0 = ex2_approx(fmaf(s[c * 32 + 2 * e], sl2, neg_mu));
            const float p1 = ex2_approx(fmaf(s[c * 32 + 2 * e + 1], sl2, neg_mu));
            l += p0 + p1;
            pk[e] = pack_bf16x2(p0, p1);
          }
          tmem_st16(tS + c * 16, pk);
        }
        // Rescale this row of O (only rows whose maximum moved; the previous
        // P V of this tile is complete because S_i(j) was committed after it).
        if (n > 0 && __any_sync(0xffffffffu, resc)) {
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t u[32];
            tmem_ld32_wait(tO + c * 32, u);
#pragma unroll
            for (int e = 0; e < 32; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * alpha);
            tmem_st32(tO + c * 32, u);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&p_full[i]);
      }
      // ---------------------------------------------------------- epilogue
      if (ok) {
        ok = mbar_wait(&o_full[i], 0, &g_prefill_status, kStatusSoftmax);
        ok = __all_sync(0xffffffffu, ok);
      }
      if (ok) {
        tc_fence_after();
        const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
        const bool store = row < N;
        const size_t orow = (static_cast<size_t>(b) * N + row) * p.Hq + h;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t u[32];
          tmem_ld32_wait(tO + c * 32, u);
          if (store) {
            if (p.o_f32) {
              float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + orow * D + c * 32);
#pragma unroll
              for (int e = 0; e < 8; ++e)
                dst[e] = make_float4(__uint_as_float(u[4 * e]) * inv_l,
                                     __uint_as_float(u[4 * e + 1]) * inv_l,
                                     __uint_as_float(u[4 * e + 2]) * inv_l,
                                     __uint_as_float(u[4 * e + 3]) * inv_l);
            } else {
              uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + orow * D +
                                                    c * 32);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                uint4 w;
                w.x = pack_bf16x2(__uint_as_float(u[8 * e + 0]) * inv_l,
                                  __uint_as_float(u[8 * e + 1]) * inv_l);
                w.y = pack_bf16x2(__uint_as_float(u[8 * e + 2]) * inv_l,
                                  __uint_as_float(u[8 * e + 3]) * inv_l);
                w.z = pack_bf16x2(__uint_as_float(u[8 * e + 4]) * inv_l,
                                  __uint_as_float(u[8 * e + 5]) * inv_l);
                w.w = pack_bf16x2(__uint_as_float(u[8 * e + 6]) * inv_l,
                                  __uint_as_float(u[8 * e + 7]) * inv_l);
                dst[e] = w;
              }
            }
          }
        }
        if (store)
          p.lse[(static_cast<size_t>(b) * p.Hq + h) * N + row] =
              (l > 0.f) ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace b300
