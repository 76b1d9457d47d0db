// Attention backward on sm_103a: dQ, dK, dV of O = softmax(scale Q K^T + mask) V
// recomputed tile by tile from the forward's saved LSE, so that, as in the
// forward, no N x N matrix reaches global memory.
//
// With P_ij = 2^(scale log2e s_ij - log2e LSE_i) (the forward's softmax weights,
// recovered exactly from the row's log-sum-exp), D_i = rowsum(dO_i * O_i):
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),  dQ = scale dS K,  dK = scale dS^T Q.
//
// Three kernels:
//   bwd_preprocess_kernel  D_i = rowsum(dO_i * O_i)                          (CUDA cores)
//   bwd_dkdv_kernel        one CTA per (sequence, kv head, 128-key tile): K_j, V_j stay
//                          in shared memory while Q_i, dO_i of every query head of the
//                          group stream through a ring; S^T = K Q^T and dP^T = V dO^T in
//                          tensor memory (keys on the lanes), P^T and dS^T written back as
//                          bf16, then dV += P^T dO and dK += dS^T Q with P^T / dS^T read
//                          from tensor memory.
//   bwd_dq_kernel          one CTA per (sequence, query head, 128-query tile): Q_i, dO_i
//                          stay, copied into tensor memory as the A operands of S and
//                          dP; K_j, V_j stream through three stages; S = Q K^T,
//                          dP = dO V^T, dS back to tensor memory, dQ += dS K.
// Splitting dQ from dK/dV recomputes S and dP once more but needs no atomics and
// gives a deterministic result.
//
// CTA layout of the two tile kernels (384 threads): warp 0 TMA producer, warp 1
// MMA issuer (whole warp, one elected lane), warp 2 tensor-memory allocator,
// warp 3 idle, warps 4-11 element-wise work in two warpgroups (one
// tensor-memory lane = one row, packed f32x2 arithmetic).
//
// Each streamed 128-row tile is handled as two halves of 64 columns, each with
// its own S and dP in tensor memory and its own element-wise warpgroup.  The
// MMA order per tile t
//   [S, dP of both halves of t issued earlier]  grad(half 0, t)  S, dP(half 0, t+1)
//   grad(half 1, t)  S, dP(half 1, t+1)
// lets one half's element-wise pass run while the tensor core works on the
// other half, as the forward does with its two query tiles.
#pragma once

#include <type_traits>

#include "ptx.cuh"

namespace b300 {

__device__ unsigned int g_bwd_status;  // OR of kStatusBwd* bits (bounded waits that ran out)
// which wait gave up (bits of g_bwd_status)
constexpr unsigned kStatusBwdProducer = 32u, kStatusBwdMma = 64u, kStatusBwdCompute = 128u,
                   kStatusBwdVec = 256u, kStatusBwdMmaP = 512u, kStatusBwdEpilogue = 1024u;

struct BwdParams {
  const void* o;          // forward output [B, N, Hq, d] (bf16 or f32: o_f32)
  const __nv_bfloat16* dO;  // [B, N, Hq, d]
  const float* lse;       // [B, Hq, N] natural log (forward)
  float* dvec;            // [B, Hq, N] rowsum(dO * O)
  void* dq;               // [B, N, Hq, d] bf16
  void* dk;               // [B, N, Hkv, d] bf16
  void* dv;               // [B, N, Hkv, d] bf16
  int B, Hq, Hkv, N;
  int causal, window, o_f32;
  float scale, scale_log2;
};

// ---------------------------------------------------------------- D = rowsum(dO * O)
// Rows are numbered in the [B, N, Hq] order of O.  A row is read by D/8 lanes,
// 16 bytes of dO (and of a bf16 O) each; a warp covers 256/D rows per pass and
// keeps kPrePasses passes of loads in flight before it reduces any of them.
constexpr int kPrePasses = 4;
template <int D>
constexpr long long bwd_preprocess_rows_per_cta() { return 8LL * (256 / D) * kPrePasses; }

__device__ __forceinline__ float dot8_bf16(const uint4& a, const uint4& b) {
  float acc = bf16lo_to_f32(a.x) * bf16lo_to_f32(b.x);
  acc = fmaf(bf16hi_to_f32(a.x), bf16hi_to_f32(b.x), acc);
  acc = fmaf(bf16lo_to_f32(a.y), bf16lo_to_f32(b.y), acc);
  acc = fmaf(bf16hi_to_f32(a.y), bf16hi_to_f32(b.y), acc);
  acc = fmaf(bf16lo_to_f32(a.z), bf16lo_to_f32(b.z), acc);
  acc = fmaf(bf16hi_to_f32(a.z), bf16hi_to_f32(b.z), acc);
  acc = fmaf(bf16lo_to_f32(a.w), bf16lo_to_f32(b.w), acc);
  acc = fmaf(bf16hi_to_f32(a.w), bf16hi_to_f32(b.w), acc);
  return acc;
}

template <int D>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const BwdParams p) {
  constexpr int LPR = D / 8;      // lanes per row
  constexpr int RPW = 32 / LPR;   // rows per warp and pass
  const int lane = threadIdx.x & 31;
  const int sub = lane / LPR, l = lane % LPR;
  const long long rows = static_cast<long long>(p.B) * p.N * p.Hq;
  const long long row0 = (static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5)) * RPW * kPrePasses;
  uint4 g[kPrePasses], o[kPrePasses], o2[kPrePasses];
#pragma unroll
  for (int u = 0; u < kPrePasses; ++u) {
    const long long row = row0 + u * RPW + sub;
    g[u] = o[u] = o2[u] = make_uint4(0u, 0u, 0u, 0u);
    if (row < rows) {
      g[u] = reinterpret_cast<const uint4*>(p.dO + row * D)[l];
      if (p.o_f32) {
        const uint4* of = reinterpret_cast<const uint4*>(static_cast<const float*>(p.o) + row * D);
        o[u] = of[2 * l];
        o2[u] = of[2 * l + 1];
      } else {
        o[u] = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.o) + row * D)[l];
      }
    }
  }
#pragma unroll
  for (int u = 0; u < kPrePasses; ++u) {
    float acc;
    if (p.o_f32) {
      const uint4 a = o[u], b = o2[u];
      acc = bf16lo_to_f32(g[u].x) * __uint_as_float(a.x);
      acc = fmaf(bf16hi_to_f32(g[u].x), __uint_as_float(a.y), acc);
      acc = fmaf(bf16lo_to_f32(g[u].y), __uint_as_float(a.z), acc);
      acc = fmaf(bf16hi_to_f32(g[u].y), __uint_as_float(a.w), acc);
      acc = fmaf(bf16lo_to_f32(g[u].z), __uint_as_float(b.x), acc);
      acc = fmaf(bf16hi_to_f32(g[u].z), __uint_as_float(b.y), acc);
      acc = fmaf(bf16lo_to_f32(g[u].w), __uint_as_float(b.z), acc);
      acc = fmaf(bf16hi_to_f32(g[u].w), __uint_as_float(b.w), acc);
    } else {
      acc = dot8_bf16(g[u], o[u]);
    }
#pragma unroll
    for (int m = LPR / 2; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
    const long long row = row0 + u * RPW + sub;
    if (l == 0 && row < rows) {
      const int h = static_cast<int>(row % p.Hq);
      const long long bi = row / p.Hq;
      const int i = static_cast<int>(bi % p.N);
      const int b = static_cast<int>(bi / p.N);
      p.dvec[(static_cast<long long>(b) * p.Hq + h) * p.N + i] = acc;
    }
  }
}

// Query row q sees key k (same rule as the forward).
__device__ __forceinline__ bool bwd_visible(int q, int k, int N, bool causal, int window) {
  if (q >= N || k >= N) return false;
  if (causal && k > q) return false;
  if (window >= 0) {
    if (q - k > window) return false;
    if (!causal && k - q > window) return false;
  }
  return true;
}

// CTA x of a grid of nt tiles x BH heads: heads in groups of kBwdHeadGroup,
// tile-major inside a group (tile index t, head index bh).
constexpr int kBwdHeadGroup = 8;
__device__ __forceinline__ void bwd_order(unsigned x, int nt, int BH, int& t, int& bh) {
  const int per = kBwdHeadGroup * nt;
  const int g = static_cast<int>(x / per);
  const int gbase = g * kBwdHeadGroup;
  const int gsz = min(kBwdHeadGroup, BH - gbase);
  const int r = static_cast<int>(x - static_cast<unsigned>(g) * per);
  t = r / gsz;
  bh = gbase + r % gsz;
}

template <int D>
struct BwdCfg {
  static constexpr int TILE = 128;                  // rows of a Q, dO, K or V tile
  static constexpr int DCH = D / 64;                // 128-byte swizzle atoms across d
  static constexpr int TILE_BYTES = TILE * D * 2;
  static constexpr int STAGES = 2;
  static constexpr int THREADS = 384;
  static constexpr int EW_THREADS = 256;  // element-wise threads (two warpgroups)
};

// ---------------------------------------------------------------- dK, dV
template <int D>
struct DkdvSmem {
  using C = BwdCfg<D>;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = C::TILE_BYTES;
  static constexpr int RING_OFF = 2 * C::TILE_BYTES;              // stage: Q tile, dO tile
  static constexpr int STAGE_BYTES = 2 * C::TILE_BYTES;
  // [2 slots][2 warpgroups][-LSE2, -D][64 queries] f32
  static constexpr int VEC_OFF = RING_OFF + C::STAGES * STAGE_BYTES;
  static constexpr int BAR_OFF = VEC_OFF + 2 * 2 * 128 * 4;
  static constexpr int BYTES = BAR_OFF + 256 + 1024;  // barriers + TMEM address, alignment slack
};

template <int D>
__global__ void __launch_bounds__(384, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const BwdParams p) {
  using C = BwdCfg<D>;
  using L = DkdvSmem<D>;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  float* vec = reinterpret_cast<float*>(smem + L::VEC_OFF);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* kv_full = bars;                // K_j, V_j landed
  uint64_t* ring_full = bars + 1;          // [STAGES]
  uint64_t* ring_empty = ring_full + STAGES;
  uint64_t* s_full = ring_empty + STAGES;  // [2] S^T and dP^T of query half w in tensor memory
  uint64_t* p_ready = s_full + 2;          // [2] P^T, dS^T of half w written (128 threads)
  uint64_t* acc_done = p_ready + 2;        // every MMA done
  uint64_t* vec_full = acc_done + 1;       // [2 slots][2 warpgroups] vectors staged (128 threads)
  uint64_t* p_half = vec_full + 4;        // [2] first 32 queries of half w written (128 threads)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(p_half + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = p.N;
  const int nkt = (N + 127) / 128;
  // Launch order: (sequence, kv head) pairs in groups of kBwdHeadGroup; within
  // a group, key tile by key tile from the first (under a causal mask the
  // first key tiles are seen by the most query tiles: heaviest CTAs first), so
  // the CTAs resident at one time share a few heads' Q and dO in L2.
  int jt, bh;
  bwd_order(blockIdx.x, nkt, p.B * p.Hkv, jt, bh);
  if (threadIdx.x == 0) B300_DCHECK(jt >= 0 && jt < nkt && bh >= 0 && bh < p.B * p.Hkv, kDbgBwdTile);
  const int hk = bh % p.Hkv;
  const int b = bh / p.Hkv;
  const int G = p.Hq / p.Hkv;
  const int c0 = jt * 128, c1 = min(c0 + 127, N - 1);
  // query rows that see at least one key of this tile
  int rlo = 0, rhi = N - 1;
  if (p.causal) rlo = c0;
  if (p.window >= 0) {
    if (!p.causal) rlo = max(0, c0 - p.window);
    rhi = min(N - 1, c1 + p.window);
  }
  const int ilo = rlo / 128, ihi = rhi / 128;
  const int nq = ihi - ilo + 1;                   // query tiles per head
  const int nsteps = G * nq;                      // (head, query tile) steps

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&ring_full[s], 1);
      mbar_init(&ring_empty[s], 1);
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(&s_full[w], 1);
      mbar_init(&p_ready[w], C::EW_THREADS / 2);
    }
    mbar_init(acc_done, 1);
    for (int x = 0; x < 4; ++x) mbar_init(&vec_full[x], C::EW_THREADS / 2);
    for (int w = 0; w < 2; ++w) mbar_init(&p_half[w], C::EW_THREADS / 2);
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // tensor memory: query half w (64 queries) has S^T at [128w, 128w+64) and dP^T
  // at [128w+64, 128w+128); dV [256,256+D)  dK [256+D,256+2D)
  const uint32_t tV = tmem + 256, tK = tmem + 256 + D;

  // Register split: launched at 168 per thread (384 x 168 = 64512); warpgroup
  // 0 (producer, MMA issuer, allocator, idle) gives back to 88 and the two
  // element-wise warpgroups take 208, so that a step's four tensor-memory
  // loads fit in registers together: 128 x 88 + 256 x 208 = 64512.
  if (warp < 4) {
  setmaxnreg_dec<88>();
  if (warp == 0) {
    // ================================================================ producer
    if (lane == 0) {
      mbar_arrive_expect_tx(kv_full, 2 * C::TILE_BYTES);
      for (int cc = 0; cc < C::DCH; ++cc) {
        tma_load_4d(smem + L::K_OFF + cc * (128 * 128), &tm_k, kv_full, cc * 64, hk, c0, b);
        tma_load_4d(smem + L::V_OFF + cc * (128 * 128), &tm_v, kv_full, cc * 64, hk, c0, b);
      }
      int t = 0;
      bool ok = true;
      for (; t < nsteps && ok; ++t) {
        const int s = t % STAGES;
        if (t >= STAGES &&
            !(ok = mbar_wait(&ring_empty[s], ((t / STAGES) - 1) & 1, &g_bwd_status,
                             kStatusBwdProducer)))
          break;
        const int h = hk * G + t / nq;
        const int r0 = (ilo + t % nq) * 128;
        uint8_t* st = smem + L::RING_OFF + s * L::STAGE_BYTES;
        mbar_arrive_expect_tx(&ring_full[s], 2 * C::TILE_BYTES);
        for (int cc = 0; cc < C::DCH; ++cc) {
          tma_load_4d(st + cc * (128 * 128), &tm_q, &ring_full[s], cc * 64, h, r0, b);
          tma_load_4d(st + C::TILE_BYTES + cc * (128 * 128), &tm_do, &ring_full[s], cc * 64, h,
                      r0, b);
        }
      }
      for (int u = max(0, t - STAGES); u < t; ++u)
        mbar_wait(&ring_full[u % STAGES], (u / STAGES) & 1, &g_bwd_status, kStatusBwdProducer);
      mbar_wait(kv_full, 0, &g_bwd_status, kStatusBwdProducer);
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    const uint32_t idS = idesc_bf16_f32(128, 64, false);  // 128 keys x 64 queries
    const uint32_t idO = idesc_bf16_f32(128, D, true);
    const uint64_t dK0 = smem_desc_sw128(smem_u32(smem + L::K_OFF), 16, 1024);
    const uint64_t dV0 = smem_desc_sw128(smem_u32(smem + L::V_OFF), 16, 1024);
    const uint64_t dR0 = smem_desc_sw128(smem_u32(smem + L::RING_OFF), 16, 1024);
    const uint64_t dRmn = smem_desc_sw128(smem_u32(smem + L::RING_OFF), 128 * 128, 1024);
    auto wait = [&](uint64_t* bar, uint32_t parity, unsigned site) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, &g_bwd_status, site));
    };
    // S^T_w = K Q_w^T and dP^T_w = V dO_w^T for query half w: rows 64w.. of the
    // stage's Q / dO tiles, 8 KB into each 128-byte-wide block (a whole number
    // of 1 KB swizzle atoms)
    auto issue_sdp = [&](int w, int s) {
      const uint64_t qK = dR0 + static_cast<uint64_t>((s * L::STAGE_BYTES + w * 64 * 128) >> 4);
      const uint64_t doK = qK + static_cast<uint64_t>(C::TILE_BYTES >> 4);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = ((kk >> 2) * (128 * 128) + (kk & 3) * 32) >> 4;
        umma_ss_warp(tmem + 128 * w, dK0 + off, qK + off, idS, kk > 0 ? 1u : 0u);
      }
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = ((kk >> 2) * (128 * 128) + (kk & 3) * 32) >> 4;
        umma_ss_warp(tmem + 128 * w + 64, dV0 + off, doK + off, idS, kk > 0 ? 1u : 0u);
      }
      umma_commit_warp(&s_full[w]);
    };
    // dV += P^T_w dO_w and dK += dS^T_w Q_w: A from tensor memory (the half's
    // bf16 pairs, in the first 32 columns of its S^T / dP^T), B the stage's
    // dO / Q rows of the half read MN-major, 16 queries per instruction.
    // Part 0 covers the half's first 32 queries (its first element-wise
    // chunk), part 1 the other 32.
    auto issue_grad = [&](int w, int s, bool first, int part) {
      const uint64_t qMN = dRmn + static_cast<uint64_t>((s * L::STAGE_BYTES) >> 4);
      const uint64_t doMN = qMN + static_cast<uint64_t>(C::TILE_BYTES >> 4);
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const int k4 = 2 * part + x;
        umma_ts_warp(tV, tmem + 128 * w + k4 * 8, doMN + (((4 * w + k4) * 16 * 128) >> 4), idO,
                     (!first || k4 > 0) ? 1u : 0u);
      }
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const int k4 = 2 * part + x;
        umma_ts_warp(tK, tmem + 128 * w + 64 + k4 * 8, qMN + (((4 * w + k4) * 16 * 128) >> 4),
                     idO, (!first || k4 > 0) ? 1u : 0u);
      }
    };
    // both parts of half w's gradients, each once the element-wise pass has
    // written its chunk
    auto grads = [&](int w, int s, bool first, uint32_t parity) {
      if (!wait(&p_half[w], parity, kStatusBwdMmaP)) return false;
      tc_fence_after();
      issue_grad(w, s, first, 0);
      if (!wait(&p_ready[w], parity, kStatusBwdMmaP)) return false;
      tc_fence_after();
      issue_grad(w, s, first, 1);
      return true;
    };
    bool ok = wait(kv_full, 0, kStatusBwdMma);
    if (ok && nsteps > 0 && (ok = wait(&ring_full[0], 0, kStatusBwdMma))) {
      tc_fence_after();
      issue_sdp(0, 0);
      issue_sdp(1, 0);
    }
    for (int t = 0; t < nsteps && ok; ++t) {
      const int s = t % STAGES, s1 = (t + 1) % STAGES;
      const bool has_next = t + 1 < nsteps;
      if (!(ok = grads(0, s, t == 0, t & 1))) break;
      if (has_next) {
        if (!(ok = wait(&ring_full[s1], ((t + 1) / STAGES) & 1, kStatusBwdMma))) break;
        tc_fence_after();
        issue_sdp(0, s1);
      }
      if (!(ok = grads(1, s, false, t & 1))) break;
      umma_commit_warp(&ring_empty[s]);
      if (has_next) issue_sdp(1, s1);
    }
    umma_commit_warp(acc_done);
    wait(acc_done, 0, kStatusBwdMma);
  }
  } else {
    setmaxnreg_inc<208>();
    // ================================================================ element-wise
    const int quarter = warp & 3;
    const int wg = (warp - 4) >> 2;     // query half: columns 64*wg .. 64*wg+63 of the tile
    const int r = quarter * 32 + lane;  // key row of this thread within the tile
    const int key = c0 + r;
    const uint32_t tS = tmem + 128 * wg, tP = tS + 64;  // this half's S^T and dP^T
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float sl2 = p.scale_log2;
    const float2 sl2x2 = make_float2(sl2, sl2);
    const bool causal = p.causal != 0;
    // this thread's entry of step t's per-query vectors for its warpgroup's
    // 64 queries, negated: -LSE (base 2) from threads 0-63, -D from threads
    // 64-127; loaded one step ahead
    auto vec_entry = [&](int t) -> float {
      const int q = (ilo + t % nq) * 128 + 64 * wg + (r & 63);
      const size_t vi = (static_cast<size_t>(b) * p.Hq + hk * G + t / nq) * N + q;
      if (q >= N) return 0.f;
      return r < 64 ? -p.lse[vi] * kLog2e : -p.dvec[vi];
    };
    float v_next = nsteps > 0 ? vec_entry(0) : 0.f;
    bool ok = true;
    for (int t = 0; t < nsteps && ok; ++t) {
      const int r0 = (ilo + t % nq) * 128;
      // the step's vectors are staged in shared memory, per warpgroup (two
      // slots; a slot is rewritten only after every thread of the warpgroup
      // has arrived for the step in between, i.e. finished reading it), so
      // the two warpgroups never wait for each other
      float* nlse = vec + ((t & 1) * 2 + wg) * 128;
      float* ndv = nlse + 64;
      (r < 64 ? nlse : ndv)[r & 63] = v_next;
      if (t + 1 < nsteps) v_next = vec_entry(t + 1);
      uint64_t* vf = &vec_full[(t & 1) * 2 + wg];
      mbar_arrive(vf);
      ok = __all_sync(0xffffffffu, mbar_wait(vf, (t >> 1) & 1, &g_bwd_status, kStatusBwdVec));
      if (!ok) break;
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[wg], t & 1, &g_bwd_status,
                                             kStatusBwdCompute));
      if (!ok) break;
      tc_fence_after();
      const bool full_tile = (r0 + 127 < N) && (c0 + 127 < N) &&
                             (!causal || r0 >= c0 + 127) &&
                             (p.window < 0 || (r0 + 127 - c0 <= p.window &&
                                               (causal || c0 + 127 - r0 <= p.window)));
      // two chunks of 32 columns, all four loads in flight behind one wait;
      // chunk ch's bf16 pairs go to columns [16ch, 16ch+16) of the same
      // array, read before any store
      uint32_t us2[2][32], ud2[2][32];
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        tmem_ld32(tS + lane_off + ch * 32, us2[ch]);
        tmem_ld32(tP + lane_off + ch * 32, ud2[ch]);
      }
      tmem_wait_ld();
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        reg_fence(us2[ch]);
        reg_fence(ud2[ch]);
      }
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        const uint32_t (&us)[32] = us2[ch];
        const uint32_t (&ud)[32] = ud2[ch];
        uint32_t pk[16], dk[16];
        // The mask test is taken once per chunk, outside the unrolled loop, so
        // that each version of the loop is one basic block whose eight
        // iterations the compiler can interleave (a branch inside the loop
        // would serialise their load -> ex2 -> pack chains).
        auto pass = [&](auto masked) {
#pragma unroll
          for (int e = 0; e < 16; e += 2) {  // four query columns per iteration
            const int col = ch * 32 + 2 * e;  // within the warpgroup's 64 queries
            const float4 nl = *reinterpret_cast<const float4*>(nlse + col);
            const float4 nd = *reinterpret_cast<const float4*>(ndv + col);
            const float2 x0 = ffma2(make_float2(__uint_as_float(us[2 * e]), __uint_as_float(us[2 * e + 1])),
                                    sl2x2, make_float2(nl.x, nl.y));
            const float2 x1 = ffma2(make_float2(__uint_as_float(us[2 * e + 2]), __uint_as_float(us[2 * e + 3])),
                                    sl2x2, make_float2(nl.z, nl.w));
            float2 p0 = make_float2(ex2_approx(x0.x), ex2_approx(x0.y));
            float2 p1 = make_float2(ex2_approx(x1.x), ex2_approx(x1.y));
            if constexpr (decltype(masked)::value) {
              const int q = r0 + 64 * wg + col;
              p0.x = bwd_visible(q, key, N, causal, p.window) ? p0.x : 0.f;
              p0.y = bwd_visible(q + 1, key, N, causal, p.window) ? p0.y : 0.f;
              p1.x = bwd_visible(q + 2, key, N, causal, p.window) ? p1.x : 0.f;
              p1.y = bwd_visible(q + 3, key, N, causal, p.window) ? p1.y : 0.f;
            }
            const float2 d0 = fadd2(make_float2(__uint_as_float(ud[2 * e]), __uint_as_float(ud[2 * e + 1])),
                                    make_float2(nd.x, nd.y));
            const float2 d1 = fadd2(make_float2(__uint_as_float(ud[2 * e + 2]), __uint_as_float(ud[2 * e + 3])),
                                    make_float2(nd.z, nd.w));
            const float2 ds0 = fmul2(p0, d0), ds1 = fmul2(p1, d1);
            pk[e] = pack_bf16x2(p0.x, p0.y);
            pk[e + 1] = pack_bf16x2(p1.x, p1.y);
            dk[e] = pack_bf16x2(ds0.x, ds0.y);
            dk[e + 1] = pack_bf16x2(ds1.x, ds1.y);
          }
        };
        if (full_tile)
          pass(std::false_type{});
        else
          pass(std::true_type{});
        tmem_st16(tS + lane_off + ch * 16, pk);
        tmem_st16(tP + lane_off + ch * 16, dk);
        // the first 32 queries' P^T and dS^T are in place: their gradient
        // MMAs may start while the second chunk is computed
        if (ch == 0) {
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&p_half[wg]);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_ready[wg]);
    }
    // ---------------------------------------------------------- epilogue
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(acc_done, 0, &g_bwd_status, kStatusBwdEpilogue));
    if (ok) {
      tc_fence_after();
      // every lane takes part in the (warp-collective) tensor-memory loads;
      // only rows inside the sequence are stored
      const size_t orow = (static_cast<size_t>(b) * N + min(key, N - 1)) * p.Hkv + hk;
      {
        const int which = wg;  // warpgroup 1 stores dV, warpgroup 2 dK
        const uint32_t tA = (which ? tK : tV) + lane_off;
        const float mul = which ? p.scale : 1.f;
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(which ? p.dk : p.dv) + orow * D;
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t u[32];
          tmem_ld32_wait(tA + cc * 32, u);
          if (key < N) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + cc * 32);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              uint4 w;
              w.x = pack_bf16x2(__uint_as_float(u[8 * e + 0]) * mul, __uint_as_float(u[8 * e + 1]) * mul);
              w.y = pack_bf16x2(__uint_as_float(u[8 * e + 2]) * mul, __uint_as_float(u[8 * e + 3]) * mul);
              w.z = pack_bf16x2(__uint_as_float(u[8 * e + 4]) * mul, __uint_as_float(u[8 * e + 5]) * mul);
              w.w = pack_bf16x2(__uint_as_float(u[8 * e + 6]) * mul, __uint_as_float(u[8 * e + 7]) * mul);
              d4[e] = w;
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------- dQ
// Three K/V stages (K tile, V tile each).  Q_i and dO_i land in stage 0's
// space and are copied into tensor memory at the start; step t loads stage
// (t + 1) mod 3, so stage 0 is first reused at step 2, once the copy is done.
template <int D>
struct DqSmem {
  using C = BwdCfg<D>;
  static constexpr int STAGES = 3;
  static constexpr int Q_OFF = 0;
  static constexpr int DO_OFF = C::TILE_BYTES;
  static constexpr int RING_OFF = 0;
  static constexpr int STAGE_BYTES = 2 * C::TILE_BYTES;
  static constexpr int BAR_OFF = RING_OFF + STAGES * STAGE_BYTES;
  static constexpr int BYTES = BAR_OFF + 256 + 1024;
  // ring stage of step t; the stage's uses before step t number t / STAGES
  static __device__ __forceinline__ int stage(int t) { return (t + 1) % STAGES; }
};

template <int D>
__global__ void __launch_bounds__(384, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const BwdParams p) {
  using C = BwdCfg<D>;
  using L = DqSmem<D>;
  constexpr int STAGES = L::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* q_full = bars;                 // Q_i, dO_i landed
  uint64_t* ring_full = bars + 1;          // [STAGES]
  uint64_t* ring_empty = ring_full + STAGES;
  uint64_t* s_full = ring_empty + STAGES;  // [2] S and dP of key half w in tensor memory
  uint64_t* p_ready = s_full + 2;          // [2] dS of half w written (128 threads)
  uint64_t* acc_done = p_ready + 2;
  uint64_t* qin_full = acc_done + 1;       // Q_i, dO_i copied into tensor memory (256 threads)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(qin_full + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = p.N;
  const int nqt = (N + 127) / 128;
  // Launch order as for dK/dV (groups of heads, tile by tile within a group),
  // from the last query tile: under a causal mask it sees the most key tiles.
  int it, bh;
  bwd_order(blockIdx.x, nqt, p.B * p.Hq, it, bh);
  if (threadIdx.x == 0) B300_DCHECK(it >= 0 && it < nqt && bh >= 0 && bh < p.B * p.Hq, kDbgBwdTile);
  if (p.causal) it = nqt - 1 - it;
  const int h = bh % p.Hq;
  const int b = bh / p.Hq;
  const int hk = h / (p.Hq / p.Hkv);
  const int r0 = it * 128, r1 = min(r0 + 127, N - 1);
  const int klo = (p.window >= 0) ? max(0, r0 - p.window) : 0;
  const int khi = p.causal ? r1 : ((p.window >= 0) ? min(N - 1, r1 + p.window) : N - 1);
  const int jlo = klo / 128, jhi = khi / 128;
  const int nsteps = jhi - jlo + 1;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&ring_full[s], 1);
      mbar_init(&ring_empty[s], 1);
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(&s_full[w], 1);
      mbar_init(&p_ready[w], C::EW_THREADS / 2);
    }
    mbar_init(acc_done, 1);
    mbar_init(qin_full, C::EW_THREADS);
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // tensor memory: key half w (64 keys) has S at [128w, 128w+64) and dP at
  // [128w+64, 128w+128); dQ [256,256+D); Q_i and dO_i as bf16 pairs (the A
  // operands of S and dP) at [384, 384+D/2) and [448, 448+D/2)
  const uint32_t tQ = tmem + 256;
  const uint32_t tQin = tmem + 384, tDOin = tmem + 448;

  // Register split as in the dK/dV kernel: 128 x 88 + 256 x 208 = 384 x 168.
  if (warp < 4) {
  setmaxnreg_dec<88>();
  if (warp == 0) {
    // ================================================================ producer
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, 2 * C::TILE_BYTES);
      for (int cc = 0; cc < C::DCH; ++cc) {
        tma_load_4d(smem + L::Q_OFF + cc * (128 * 128), &tm_q, q_full, cc * 64, h, r0, b);
        tma_load_4d(smem + L::DO_OFF + cc * (128 * 128), &tm_do, q_full, cc * 64, h, r0, b);
      }
      int t = 0;
      bool ok = true;
      for (; t < nsteps && ok; ++t) {
        const int s = L::stage(t);
        if (t >= STAGES &&
            !(ok = mbar_wait(&ring_empty[s], ((t / STAGES) - 1) & 1, &g_bwd_status,
                             kStatusBwdProducer)))
          break;
        // stage 0 holds Q_i and dO_i until they are in tensor memory
        if (t == STAGES - 1 &&
            !(ok = mbar_wait(qin_full, 0, &g_bwd_status, kStatusBwdProducer)))
          break;
        const int c0 = (jlo + t) * 128;
        uint8_t* st = smem + L::RING_OFF + s * L::STAGE_BYTES;
        mbar_arrive_expect_tx(&ring_full[s], 2 * C::TILE_BYTES);
        for (int cc = 0; cc < C::DCH; ++cc) {
          tma_load_4d(st + cc * (128 * 128), &tm_k, &ring_full[s], cc * 64, hk, c0, b);
          tma_load_4d(st + C::TILE_BYTES + cc * (128 * 128), &tm_v, &ring_full[s], cc * 64, hk,
                      c0, b);
        }
      }
      for (int u = max(0, t - STAGES); u < t; ++u)
        mbar_wait(&ring_full[L::stage(u)], (u / STAGES) & 1, &g_bwd_status, kStatusBwdProducer);
      mbar_wait(q_full, 0, &g_bwd_status, kStatusBwdProducer);
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    const uint32_t idS = idesc_bf16_f32(128, 64, false);  // 128 queries x 64 keys
    const uint32_t idO = idesc_bf16_f32(128, D, true);
    const uint64_t dR0 = smem_desc_sw128(smem_u32(smem + L::RING_OFF), 16, 1024);
    const uint64_t dRmn = smem_desc_sw128(smem_u32(smem + L::RING_OFF), 128 * 128, 1024);
    auto wait = [&](uint64_t* bar, uint32_t parity, unsigned site) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, &g_bwd_status, site));
    };
    // S_w = Q K_w^T and dP_w = dO V_w^T for key half w: rows 64w.. of the
    // stage's K / V tiles (8 KB into each 128-byte-wide block)
    // Q and dO are read from tensor memory (8 columns = 16 elements of d per
    // instruction), so that shared memory serves only the K / V half (2 KB
    // per instruction instead of 6 KB with Q and dO there too).
    auto issue_sdp = [&](int w, int s) {
      const uint64_t kK = dR0 + static_cast<uint64_t>((s * L::STAGE_BYTES + w * 64 * 128) >> 4);
      const uint64_t vK = kK + static_cast<uint64_t>(C::TILE_BYTES >> 4);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = ((kk >> 2) * (128 * 128) + (kk & 3) * 32) >> 4;
        umma_ts_warp(tmem + 128 * w, tQin + kk * 8, kK + off, idS, kk > 0 ? 1u : 0u);
      }
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = ((kk >> 2) * (128 * 128) + (kk & 3) * 32) >> 4;
        umma_ts_warp(tmem + 128 * w + 64, tDOin + kk * 8, vK + off, idS, kk > 0 ? 1u : 0u);
      }
      umma_commit_warp(&s_full[w]);
    };
    // dQ += dS_w K_w: dS (bf16 pairs in the first 32 columns of the half's dP)
    // from tensor memory, the stage's K rows of the half read MN-major
    auto issue_grad = [&](int w, int s, bool first) {
      const uint64_t kMN = dRmn + static_cast<uint64_t>((s * L::STAGE_BYTES) >> 4);
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4)
        umma_ts_warp(tQ, tmem + 128 * w + 64 + k4 * 8, kMN + (((4 * w + k4) * 16 * 128) >> 4),
                     idO, (!first || k4 > 0) ? 1u : 0u);
    };
    bool ok = wait(qin_full, 0, kStatusBwdMma);
    if (ok && nsteps > 0 && (ok = wait(&ring_full[L::stage(0)], 0, kStatusBwdMma))) {
      tc_fence_after();
      issue_sdp(0, L::stage(0));
      issue_sdp(1, L::stage(0));
    }
    for (int t = 0; t < nsteps && ok; ++t) {
      const int s = L::stage(t), s1 = L::stage(t + 1);
      const bool has_next = t + 1 < nsteps;
      if (!(ok = wait(&p_ready[0], t & 1, kStatusBwdMmaP))) break;
      tc_fence_after();
      issue_grad(0, s, t == 0);
      if (has_next) {
        if (!(ok = wait(&ring_full[s1], ((t + 1) / STAGES) & 1, kStatusBwdMma))) break;
        tc_fence_after();
        issue_sdp(0, s1);
      }
      if (!(ok = wait(&p_ready[1], t & 1, kStatusBwdMmaP))) break;
      tc_fence_after();
      issue_grad(1, s, false);
      umma_commit_warp(&ring_empty[s]);
      if (has_next) issue_sdp(1, s1);
    }
    umma_commit_warp(acc_done);
    wait(acc_done, 0, kStatusBwdMma);
  }
  } else {
    setmaxnreg_inc<208>();
    // ================================================================ element-wise
    const int quarter = warp & 3;
    const int wg = (warp - 4) >> 2;     // key half: columns 64*wg .. 64*wg+63 of the tile
    const int r = quarter * 32 + lane;  // query row of this thread within the tile
    const int row = r0 + r;
    const uint32_t tS = tmem + 128 * wg, tP = tS + 64;  // this half's S and dP
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float sl2 = p.scale_log2;
    const bool causal = p.causal != 0;
    const size_t vi = (static_cast<size_t>(b) * p.Hq + h) * N + row;
    const float nlse = (row < N) ? -p.lse[vi] * kLog2e : 0.f;
    const float ndrow = (row < N) ? -p.dvec[vi] : 0.f;
    const float2 sl2x2 = make_float2(sl2, sl2), nlse2 = make_float2(nlse, nlse);
    const float2 ndrow2 = make_float2(ndrow, ndrow);
    // Q_i (warpgroup 0) or dO_i (warpgroup 1) into tensor memory: this
    // thread's row, un-swizzled from the TMA tile (16-byte unit k of row r
    // at position k ^ (r mod 8)), as bf16 pairs in d order
    bool ok = __all_sync(0xffffffffu, mbar_wait(q_full, 0, &g_bwd_status, kStatusBwdCompute));
    if (ok) {
      const uint8_t* src = smem + (wg ? L::DO_OFF : L::Q_OFF) + r * 128;
#pragma unroll
      for (int cc = 0; cc < C::DCH; ++cc) {
        uint32_t w[32];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint4 v4 = *reinterpret_cast<const uint4*>(src + cc * (128 * 128) + ((k ^ (r & 7)) << 4));
          w[4 * k] = v4.x;
          w[4 * k + 1] = v4.y;
          w[4 * k + 2] = v4.z;
          w[4 * k + 3] = v4.w;
        }
        tmem_st32((wg ? tDOin : tQin) + lane_off + cc * 32, w);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(qin_full);
    }
    for (int t = 0; t < nsteps && ok; ++t) {
      const int c0 = (jlo + t) * 128;
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[wg], t & 1, &g_bwd_status,
                                             kStatusBwdCompute));
      if (!ok) break;
      tc_fence_after();
      const bool full_tile = (r0 + 127 < N) && (c0 + 127 < N) &&
                             (!causal || r0 >= c0 + 127) &&
                             (p.window < 0 || (r0 + 127 - c0 <= p.window &&
                                               (causal || c0 + 127 - r0 <= p.window)));
      // two chunks of 32 columns, all four loads behind one wait; chunk ch's
      // bf16 pairs go to columns [16ch, 16ch+16) of the half's dP, read
      // before any store
      uint32_t us2[2][32], ud2[2][32];
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        tmem_ld32(tS + lane_off + ch * 32, us2[ch]);
        tmem_ld32(tP + lane_off + ch * 32, ud2[ch]);
      }
      tmem_wait_ld();
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        reg_fence(us2[ch]);
        reg_fence(ud2[ch]);
      }
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        const uint32_t (&us)[32] = us2[ch];
        const uint32_t (&ud)[32] = ud2[ch];
        uint32_t dk[16];
        // the mask test outside the unrolled loop (see the dK/dV kernel)
        auto pass = [&](auto masked) {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 x = ffma2(make_float2(__uint_as_float(us[2 * e]), __uint_as_float(us[2 * e + 1])),
                                   sl2x2, nlse2);
            float2 pe = make_float2(ex2_approx(x.x), ex2_approx(x.y));
            if constexpr (decltype(masked)::value) {
              const int key = c0 + 64 * wg + ch * 32 + 2 * e;
              pe.x = bwd_visible(row, key, N, causal, p.window) ? pe.x : 0.f;
              pe.y = bwd_visible(row, key + 1, N, causal, p.window) ? pe.y : 0.f;
            }
            const float2 dd = fadd2(make_float2(__uint_as_float(ud[2 * e]), __uint_as_float(ud[2 * e + 1])),
                                    ndrow2);
            const float2 ds = fmul2(pe, dd);
            dk[e] = pack_bf16x2(ds.x, ds.y);
          }
        };
        if (full_tile)
          pass(std::false_type{});
        else
          pass(std::true_type{});
        tmem_st16(tP + lane_off + ch * 16, dk);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_ready[wg]);
    }
    // ---------------------------------------------------------- epilogue
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(acc_done, 0, &g_bwd_status, kStatusBwdEpilogue));
    if (ok) {
      tc_fence_after();
      // every lane takes part in the (warp-collective) tensor-memory loads;
      // only rows inside the sequence are stored
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.dq) +
                           ((static_cast<size_t>(b) * N + min(row, N - 1)) * p.Hq + h) * D;
#pragma unroll 1
      for (int cc = wg * (D / 64); cc < (wg + 1) * (D / 64); ++cc) {  // half of d per warpgroup
        uint32_t u[32];
        tmem_ld32_wait(tQ + lane_off + cc * 32, u);
        if (row >= N) continue;
        uint4* d4 = reinterpret_cast<uint4*>(dst + cc * 32);
        const float mul = p.scale;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(u[8 * e + 0]) * mul, __uint_as_float(u[8 * e + 1]) * mul);
          w.y = pack_bf16x2(__uint_as_float(u[8 * e + 2]) * mul, __uint_as_float(u[8 * e + 3]) * mul);
          w.z = pack_bf16x2(__uint_as_float(u[8 * e + 4]) * mul, __uint_as_float(u[8 * e + 5]) * mul);
          w.w = pack_bf16x2(__uint_as_float(u[8 * e + 6]) * mul, __uint_as_float(u[8 * e + 7]) * mul);
          d4[e] = w;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace b300
