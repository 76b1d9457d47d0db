// Split-KV single-query decode and the logsumexp tree combine, sm_103a.
//
// The key axis of every sequence is cut into chunks; one CTA per (sequence,
// kv head, chunk) computes, for every query head of the GQA group, the
// partial triple over its keys
//     m = max_j s_j,  l = sum_j 2^(s_j - m),  o = sum_j 2^(s_j - m) v_j
// (scores in base-2 units inside the kernel; m is stored in natural-log
// units).  A second kernel merges the triples of a row with the associative
//     (m,l,o) + (m',l',o') = (M, l 2^(m-M) + l' 2^(m'-M), o 2^(m-M) + o' 2^(m'-M))
// in a tree.  Source: "Tree Attention: Topology-aware Decoding for
// Long-Context Attention on GPU Clusters" (express24.ir), abstract -- the
// reduction across the sequence axis is associative and parallel as a tree;
// here the tree runs inside one GPU.
//
// The decode path is bound by HBM bandwidth: each K/V byte is read once for
// the whole GQA group (the inter-head packing idea of "FlashAttention for
// Scalable Vector Architectures", gist.science), staged by TMA into a shared
// memory ring, and read back with 128-bit loads.  Dot products run on CUDA
// cores with a butterfly reduce-scatter across the lanes that share a key.
#pragma once

#include <type_traits>

#include "ptx.cuh"

namespace b300 {

__device__ unsigned int g_decode_status;

constexpr unsigned kStatusDecodeProducer = 8u, kStatusDecodeConsumer = 16u;
// A paged decode met a block-table entry outside [0, num_pages): that stage
// was treated as holding no keys (an input error, not a timeout).
constexpr unsigned kStatusDecodeBadPage = 2048u;

constexpr int kDecSub = 64;      // keys per ring stage
constexpr int kDecCWarps = 4;    // consumer warps (16 keys of each stage each)
constexpr int kDecThreads = 160; // + one producer warp

struct DecodeParams {
  const __nv_bfloat16* q;  // [B, Hq, D]
  const int* kv_len;       // [B]
  float* part_m;           // [B*Hq, S]   natural-log units
  float* part_l;           // [B*Hq, S]
  float* part_o;           // [B*Hq, S, D]
  float* seg_m;            // [B*Hq, nseg]  second level of the merge (S > 64)
  float* seg_l;            // [B*Hq, nseg]
  float* seg_o;            // [B*Hq, nseg, D]
  int B, Hq, Hkv, Lmax, chunk, S, G;
  float scale_log2;
  // Paged cache (block_table != NULL): K/V are [num_pages, page_size, Hkv, D]
  // and logical key k of sequence b lives in physical page
  // block_table[b * pages_per_seq + k / page_size], row k % page_size.
  // page_size is a multiple of the 64-key stage, so a stage never straddles pages.
  const int* block_table;
  int page_size, pages_per_seq, num_pages;
};

template <int D>
struct DecCfg {
  // Two 64-key stages per CTA at d=128 (four at d=64) keep the ring at 64 KB,
  // so that three CTAs share an SM and their streams overlap one another's
  // start and end.
  static constexpr int STAGES = (D == 128) ? 2 : 4;
  static constexpr int HALF_BYTES = kDecSub * D * 2;  // K (or V) rows of one stage
  static constexpr int STAGE_BYTES = 2 * HALF_BYTES;
  static constexpr int LPK = D / 8;          // lanes that share one key row (16 B each)
  static constexpr int NG = 32 / LPK;        // key groups per warp
  static constexpr int KPG = 16 / NG;        // keys per group per stage
  static constexpr int STEPS = (LPK == 16) ? 4 : 3;  // log2(LPK)
};

template <int D, int GT>
struct DecSmem {
  static constexpr int RING = DecCfg<D>::STAGES * DecCfg<D>::STAGE_BYTES;
  static constexpr int SCORES = kDecCWarps * 16 * GT * 4;            // per-warp scores
  static constexpr int PROBS = kDecCWarps * 16 * GT * 8;             // per-warp (p, p) pairs
  static constexpr int MERGE_O = kDecCWarps * GT * D * 4;            // per-warp o (aliases the ring)
  static constexpr int MERGE_ML = 2 * kDecCWarps * GT * 4;           // per-warp m, l
  static constexpr int BARS = 2 * DecCfg<D>::STAGES * 8;
  static_assert(MERGE_O <= RING, "the merge buffer reuses the drained ring");
  static constexpr int OFF_SCORES = RING;
  static constexpr int OFF_PROBS = OFF_SCORES + SCORES;
  static constexpr int OFF_ML = OFF_PROBS + PROBS;
  static constexpr int OFF_BARS = (OFF_ML + MERGE_ML + 15) & ~15;
  // ints: [0, STAGES) "stage holds keys" flags written by the producer,
  // [STAGES] "a consumer wait ran out" flag
  static constexpr int OFF_FLAGS = OFF_BARS + BARS;
  static constexpr int FLAGS = (DecCfg<D>::STAGES + 1) * 4;
  static constexpr int BYTES = OFF_FLAGS + FLAGS + 128;  // + alignment slack
};

// Eight bf16 (one 16-byte load) as four f32 pairs.
__device__ __forceinline__ void unpack8(const uint4 w, float2 (&f)[4]) {
  f[0] = make_float2(bf16lo_to_f32(w.x), bf16hi_to_f32(w.x));
  f[1] = make_float2(bf16lo_to_f32(w.y), bf16hi_to_f32(w.y));
  f[2] = make_float2(bf16lo_to_f32(w.z), bf16hi_to_f32(w.z));
  f[3] = make_float2(bf16lo_to_f32(w.w), bf16hi_to_f32(w.w));
}

// One CTA: (split = blockIdx.x, kv head x head group = blockIdx.y, sequence = blockIdx.z).
// GT query heads per CTA (the whole GQA group when it is 1, 2, 4 or 8 heads).
// Arithmetic on f32 pairs (fma.rn.f32x2) halves the instruction count of the
// dot products and of the P V accumulation, which keeps the kernel on the
// memory roofline instead of the issue rate.
template <int D, int GT>
__global__ void __launch_bounds__(kDecThreads, (GT <= 4) ? 3 : 1)
    decode_partial_kernel(const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const DecodeParams p) {
  using C = DecCfg<D>;
  using L = DecSmem<D, GT>;
  constexpr int STAGES = C::STAGES;
  constexpr int LPK = C::LPK, KPG = C::KPG;
  constexpr int VAL = KPG * GT;  // partial dot products per lane before the reduce-scatter

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                             ~static_cast<uintptr_t>(127));
  float* s_sm = reinterpret_cast<float*>(smem + L::OFF_SCORES);
  float2* p_sm = reinterpret_cast<float2*>(smem + L::OFF_PROBS);
  float* mo_sm = reinterpret_cast<float*>(smem);  // after the last stage is consumed
  float* mm_sm = reinterpret_cast<float*>(smem + L::OFF_ML);
  float* ml_sm = mm_sm + kDecCWarps * GT;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::OFF_BARS);
  uint64_t* empty = full + STAGES;
  volatile int* stage_ok = reinterpret_cast<volatile int*>(smem + L::OFF_FLAGS);
  volatile int* failed = stage_ok + STAGES;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int split = blockIdx.x;
  const int ngroups = p.G / GT;
  const int hkv = blockIdx.y / ngroups;
  const int hq0 = hkv * p.G + (blockIdx.y % ngroups) * GT;
  const int b = blockIdx.z;

  // The tree combine that follows may launch now: it waits for this whole
  // grid's partials before reading them (griddepcontrol.wait), so its launch
  // overlaps this grid's last CTAs instead of following them.
  grid_launch_dependents();
  int len = p.kv_len[b];
  if (threadIdx.x == 0 && split == 0 && blockIdx.y == 0)
    B300_DCHECK(len >= 0 && len <= p.Lmax, kDbgKvLen);
  if (threadIdx.x == 0)
    B300_DCHECK(b < p.B && hq0 + GT <= p.Hq && split < p.S, kDbgDecodeSplit);
  len = min(max(len, 0), p.Lmax);
  const int key0 = split * p.chunk;
  const int nkeys = min(max(len - key0, 0), p.chunk);
  const int nsub = (nkeys + kDecSub - 1) / kDecSub;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kDecCWarps);
    }
    *failed = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kDecCWarps) {
    // ================================================================ producer
    if (lane == 0 && nsub > 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      int issued = 0;
      for (; issued < nsub; ++issued) {
        const int s = issued % STAGES;
        if (issued >= STAGES &&
            !mbar_wait(&empty[s], ((issued / STAGES) - 1) & 1, &g_decode_status,
                       kStatusDecodeProducer))
          break;
        uint8_t* dst = smem + s * C::STAGE_BYTES;
        const int key = key0 + issued * kDecSub;
        int c2 = key, c3 = b;  // row and outer coordinate of the [.., rows, Hkv, D] view
        bool page_ok = true;
        if (p.block_table) {
          c2 = key % p.page_size;
          c3 = p.block_table[static_cast<size_t>(b) * p.pages_per_seq + key / p.page_size];
          page_ok = c3 >= 0 && c3 < p.num_pages;
        }
        // the flag is published by the arrive below (release) and read after
        // the consumers' wait on it (acquire)
        stage_ok[s] = page_ok ? 1 : 0;
        if (page_ok) {
          mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
          tma_load_4d(dst, &tm_k, &full[s], 0, hkv, c2, c3);
          tma_load_4d(dst + C::HALF_BYTES, &tm_v, &full[s], 0, hkv, c2, c3);
        } else {
          atomicOr(&g_decode_status, kStatusDecodeBadPage);
          mbar_arrive(&full[s]);  // no copy: the stage counts as holding no keys
        }
      }
      for (int u = max(0, issued - STAGES); u < issued; ++u)
        mbar_wait(&full[u % STAGES], (u / STAGES) & 1, &g_decode_status, kStatusDecodeProducer);
    }
    return;  // the producer takes no part in the merge below
  }

  // ================================================================ consumers
  const int grp = lane / LPK;  // key group within the warp
  const int li = lane % LPK;   // 8 consecutive elements of d: [8*li, 8*li+8)
  float* s_w = s_sm + warp * 16 * GT;
  float2* p_w = p_sm + warp * 16 * GT;

  float2 qf[GT][4];  // q * scale * log2(e), this lane's slice of d, as pairs
#pragma unroll
  for (int g = 0; g < GT; ++g) {
    const uint4 w = *reinterpret_cast<const uint4*>(
        p.q + (static_cast<size_t>(b) * p.Hq + hq0 + g) * D + 8 * li);
    unpack8(w, qf[g]);
#pragma unroll
    for (int e = 0; e < 4; ++e)
      qf[g][e] = make_float2(qf[g][e].x * p.scale_log2, qf[g][e].y * p.scale_log2);
  }
  float2 acc[GT][4];
#pragma unroll
  for (int g = 0; g < GT; ++g)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[g][e] = make_float2(0.f, 0.f);
  float m_ref[GT];  // base-2 running maximum per head (warp-uniform)
#pragma unroll
  for (int g = 0; g < GT; ++g) m_ref[g] = -INFINITY;
  float lsum = 0.f;  // this lane's share of l for head (lane % GT)

  for (int sub = 0; sub < nsub; ++sub) {
    const int stage = sub % STAGES;
    bool ok = mbar_wait(&full[stage], (sub / STAGES) & 1, &g_decode_status, kStatusDecodeConsumer);
    if (!__all_sync(0xffffffffu, ok)) {
      *failed = 1;
      break;
    }
    const uint8_t* Ks = smem + stage * C::STAGE_BYTES;
    const uint8_t* Vs = Ks + C::HALF_BYTES;
    const int nvalid = stage_ok[stage] ? min(kDecSub, nkeys - sub * kDecSub) : 0;
    const int wkey0 = warp * 16;  // this warp's 16 keys of the stage

    // ---- s = q . k for KPG keys x GT heads, partial over this lane's 8 elements
    float val[VAL];
#pragma unroll
    for (int kk = 0; kk < KPG; ++kk) {
      const int key = wkey0 + grp * KPG + kk;
      float2 kf[4];
      unpack8(*reinterpret_cast<const uint4*>(Ks + key * (D * 2) + li * 16), kf);
#pragma unroll
      for (int g = 0; g < GT; ++g) {
        float2 a = fmul2(qf[g][0], kf[0]);
        a = ffma2(qf[g][1], kf[1], a);
        a = ffma2(qf[g][2], kf[2], a);
        a = ffma2(qf[g][3], kf[3], a);
        val[kk * GT + g] = a.x + a.y;
      }
    }
    // ---- butterfly reduce-scatter over the LPK lanes of the group
    int base = 0;
#pragma unroll
    for (int st = 0, cur = VAL; st < C::STEPS; ++st) {
      const int mask = LPK >> (st + 1);
      if (cur >= 2) {
        const int half = cur / 2;
        const bool up = (lane & mask) != 0;
#pragma unroll
        for (int v = 0; v < VAL / 2; ++v) {
          if (v < half) {
            const float send = up ? val[v] : val[v + half];
            const float keep = up ? val[v + half] : val[v];
            val[v] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
          }
        }
        if (up) base += half;
        cur = half;
      } else {
        val[0] += __shfl_xor_sync(0xffffffffu, val[0], mask);
      }
    }
    constexpr int FINAL = (VAL >= LPK) ? VAL / LPK : 1;
#pragma unroll
    for (int v = 0; v < FINAL; ++v) {
      const int idx = base + v;  // = key_in_group * GT + head
      s_w[(grp * KPG + idx / GT) * GT + idx % GT] = val[v];
    }
    __syncwarp();

    // ---- online softmax over the warp's 16 keys x GT heads
    constexpr int NV = (16 * GT + 31) / 32;
    const int myg = lane % GT;
    float x[NV];
    float mx = -INFINITY;
#pragma unroll
    for (int t = 0; t < NV; ++t) {
      const int v = lane + 32 * t;
      x[t] = -INFINITY;
      if (v < 16 * GT && wkey0 + v / GT < nvalid) x[t] = s_w[v];
      mx = fmaxf(mx, x[t]);
    }
#pragma unroll
    for (int mask = GT; mask < 32; mask <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, mask));
    float mu_mine = 0.f;
#pragma unroll
    for (int g = 0; g < GT; ++g) {
      const float mn = fmaxf(m_ref[g], __shfl_sync(0xffffffffu, mx, g));
      if (mn > m_ref[g] + kRescaleThreshold) {  // warp-uniform
        const float alpha = ex2_approx(m_ref[g] - mn);
        m_ref[g] = mn;
        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[g][e] = fmul2(acc[g][e], a2);
        if (myg == g) lsum *= alpha;
      }
      if (myg == g) mu_mine = (m_ref[g] == -INFINITY) ? 0.f : m_ref[g];
    }
#pragma unroll
    for (int t = 0; t < NV; ++t) {
      const int v = lane + 32 * t;
      const float pv = ex2_approx(x[t] - mu_mine);
      lsum += pv;
      if (v < 16 * GT) p_w[v] = make_float2(pv, pv);
    }
    __syncwarp();

    // ---- o += p v over this group's keys.  V rows at or past nvalid may hold
    // anything (0 times a non-finite value is not 0), so a partial stage
    // skips them; a full stage takes the unguarded loop, one basic block whose
    // keys the compiler can interleave (the test is uniform over the CTA).
    auto pv_keys = [&](auto guarded) {
#pragma unroll
      for (int kk = 0; kk < KPG; ++kk) {
        const int kl = grp * KPG + kk;
        if (!decltype(guarded)::value || wkey0 + kl < nvalid) {
          float2 vf[4];
          unpack8(*reinterpret_cast<const uint4*>(Vs + (wkey0 + kl) * (D * 2) + li * 16), vf);
#pragma unroll
          for (int g = 0; g < GT; ++g) {
            const float2 pg = p_w[kl * GT + g];
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[g][e] = ffma2(vf[e], pg, acc[g][e]);
          }
        }
      }
    };
    if (nvalid == kDecSub)
      pv_keys(std::false_type{});
    else
      pv_keys(std::true_type{});
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
  }

  // ---- merge the key groups of the warp, then the four warps.  The merge
  // buffer for o reuses the ring: every stage has landed and been consumed.
#pragma unroll
  for (int mask = LPK; mask < 32; mask <<= 1) {
#pragma unroll
    for (int g = 0; g < GT; ++g)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc[g][e].x += __shfl_xor_sync(0xffffffffu, acc[g][e].x, mask);
        acc[g][e].y += __shfl_xor_sync(0xffffffffu, acc[g][e].y, mask);
      }
  }
#pragma unroll
  for (int mask = GT; mask < 32; mask <<= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, mask);
  named_bar_sync(1, kDecCWarps * 32);  // every warp is done reading the ring
  if (*failed) {
    // A wait ran out: copies may still be landing in the ring, so it is not
    // reused.  The split gets the identity partial (-inf, 0, 0).
    for (int idx = threadIdx.x; idx < GT * D; idx += kDecCWarps * 32) {
      const int g = idx / D, dd = idx % D;
      const size_t prow = static_cast<size_t>(b) * p.Hq + hq0 + g;
      p.part_o[(prow * p.S + split) * D + dd] = 0.f;
      if (dd == 0) {
        p.part_m[prow * p.S + split] = -INFINITY;
        p.part_l[prow * p.S + split] = 0.f;
      }
    }
    return;
  }
  if (lane < LPK) {
#pragma unroll
    for (int g = 0; g < GT; ++g)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        *reinterpret_cast<float2*>(&mo_sm[(warp * GT + g) * D + 8 * lane + 2 * e]) = acc[g][e];
  }
#pragma unroll
  for (int g = 0; g < GT; ++g)
    if (lane == g) {
      mm_sm[warp * GT + g] = m_ref[g];
      ml_sm[warp * GT + g] = lsum;
    }
  named_bar_sync(1, kDecCWarps * 32);
  for (int idx = threadIdx.x; idx < GT * D; idx += kDecCWarps * 32) {
    const int g = idx / D, dd = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecCWarps; ++w) M = fmaxf(M, mm_sm[w * GT + g]);
    float o = 0.f, lt = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kDecCWarps; ++w) {
        const float mw = mm_sm[w * GT + g];
        if (mw != -INFINITY) {
          const float c = ex2_approx(mw - M);
          o = fmaf(mo_sm[(w * GT + g) * D + dd], c, o);
          lt = fmaf(ml_sm[w * GT + g], c, lt);
        }
      }
    }
    const size_t prow = static_cast<size_t>(b) * p.Hq + hq0 + g;
    p.part_o[(prow * p.S + split) * D + dd] = o;
    if (dd == 0) {
      p.part_m[prow * p.S + split] = (M == -INFINITY) ? -INFINITY : M * kLn2;
      p.part_l[prow * p.S + split] = lt;
    }
  }
}

// ---------------------------------------------------------------------------
// Tree combine.  One row's num_splits partials are cut into C contiguous
// segments (C = 1..8 CTAs, one thread-block cluster per row).  Inside a CTA,
// a lane owns four consecutive columns of d (one 16-byte load of o per
// partial; at d = 64 two partials share a warp load), and each warp takes its
// partials eight at a time: the eight loads of m, l and o are issued together
// (none depends on another), merged pairwise in three levels, and folded into
// the warp's running triple.  The NW warp triples are then merged pairwise in
// log2(NW) levels, and finally CTA 0 of the cluster merges the C CTA triples,
// read from the other CTAs' shared memory, pairwise in log2(C) levels.
// ---------------------------------------------------------------------------

constexpr int kCombBatch = 8;
constexpr int kRowsBatch = 16;
constexpr int kCombMaxCluster = 8;

struct Triple4 {
  float m, l;  // m in base-2 units
  float4 o;
};

__device__ __forceinline__ Triple4 lse_merge4(Triple4 a, Triple4 c) {
  if (c.m == -INFINITY) return a;
  if (a.m == -INFINITY) return c;
  const float M = fmaxf(a.m, c.m);
  const float wa = ex2_approx(a.m - M), wc = ex2_approx(c.m - M);
  Triple4 r;
  r.m = M;
  r.l = fmaf(a.l, wa, c.l * wc);
  r.o = make_float4(fmaf(a.o.x, wa, c.o.x * wc), fmaf(a.o.y, wa, c.o.y * wc),
                    fmaf(a.o.z, wa, c.o.z * wc), fmaf(a.o.w, wa, c.o.w * wc));
  return r;
}

// Few partials per row: one warp per row (four rows per CTA), a lane owns
// four columns of d, and the row's partials are loaded sixteen at a time (at
// d = 128 the whole row of a 16-split decode in one round trip) with no
// branch around the loads; no shared memory and no barrier.
template <int D>
__global__ void __launch_bounds__(128)
    lse_combine_rows_kernel(const float* __restrict__ pm, const float* __restrict__ pl,
                            const float* __restrict__ po, void* out, float* lse, int rows, int S,
                            int o_f32) {
  constexpr int LPS = D / 4;
  constexpr int SPW = 32 / LPS;
  grid_dependency_wait();
  const int lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int sub = lane / LPS, c4 = lane % LPS;
  const float* mrow = pm + row * S;
  const float* lrow = pl + row * S;
  const float4* orow = reinterpret_cast<const float4*>(po + row * S * D) + c4;
  Triple4 acc{-INFINITY, 0.f, make_float4(0.f, 0.f, 0.f, 0.f)};
  for (int j0 = sub; j0 < S; j0 += SPW * kRowsBatch) {
    Triple4 t[kRowsBatch];
#pragma unroll
    for (int u = 0; u < kRowsBatch; ++u) {
      const int s = min(j0 + u * SPW, S - 1);
      t[u].m = __ldg(mrow + s);
      t[u].l = __ldg(lrow + s);
      t[u].o = __ldg(orow + static_cast<size_t>(s) * (D / 4));
    }
#pragma unroll
    for (int u = 0; u < kRowsBatch; ++u)
      t[u].m = (j0 + u * SPW < S) ? t[u].m * kLog2e : -INFINITY;
#pragma unroll
    for (int w = 1; w < kRowsBatch; w <<= 1)
#pragma unroll
      for (int u = 0; u + w < kRowsBatch; u += 2 * w) t[u] = lse_merge4(t[u], t[u + w]);
    acc = lse_merge4(acc, t[0]);
  }
  if constexpr (SPW == 2) {
    Triple4 other;
    other.m = __shfl_xor_sync(0xffffffffu, acc.m, LPS);
    other.l = __shfl_xor_sync(0xffffffffu, acc.l, LPS);
    other.o.x = __shfl_xor_sync(0xffffffffu, acc.o.x, LPS);
    other.o.y = __shfl_xor_sync(0xffffffffu, acc.o.y, LPS);
    other.o.z = __shfl_xor_sync(0xffffffffu, acc.o.z, LPS);
    other.o.w = __shfl_xor_sync(0xffffffffu, acc.o.w, LPS);
    acc = sub ? lse_merge4(other, acc) : lse_merge4(acc, other);
  }
  if (sub != 0) return;
  const float inv = (acc.l > 0.f) ? 1.f / acc.l : 0.f;
  const float4 v = make_float4(acc.o.x * inv, acc.o.y * inv, acc.o.z * inv, acc.o.w * inv);
  const size_t oi = static_cast<size_t>(row) * D + 4 * c4;
  if (o_f32) {
    *reinterpret_cast<float4*>(static_cast<float*>(out) + oi) = v;
  } else {
    uint2 w;
    w.x = pack_bf16x2(v.x, v.y);
    w.y = pack_bf16x2(v.z, v.w);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + oi) = w;
  }
  if (c4 == 0) lse[row] = (acc.l > 0.f) ? (acc.m + __log2f(acc.l)) * kLn2 : -INFINITY;
}

// First level of the two-level merge used by the decode (which has workspace
// for it): CTA (segment, row) merges partials [64 seg, 64 seg + 64) of its
// row -- four warps, sixteen partials each at d = 128, loaded eight at a time
// -- and writes the segment's triple (m in natural-log units, like a partial)
// to the second-level arrays, which lse_combine_rows_kernel then merges.
constexpr int kCombSeg = 64;

template <int D>
__global__ void __launch_bounds__(128)
    lse_combine_segments_kernel(const float* __restrict__ pm, const float* __restrict__ pl,
                                const float* __restrict__ po, float* m2, float* l2, float* o2,
                                int S, int nseg) {
  constexpr int LPS = D / 4;
  constexpr int SPW = 32 / LPS;
  constexpr int NW = 4;
  __shared__ Triple4 red[NW][LPS];
  grid_dependency_wait();
  const int seg = blockIdx.x;
  const long long row = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane / LPS, c4 = lane % LPS;
  const int sb = seg * kCombSeg, se = min(S, sb + kCombSeg);
  const float* mrow = pm + row * S;
  const float* lrow = pl + row * S;
  const float4* orow = reinterpret_cast<const float4*>(po + row * S * D) + c4;
  Triple4 acc{-INFINITY, 0.f, make_float4(0.f, 0.f, 0.f, 0.f)};
  constexpr int STRIDE = NW * SPW;
  for (int j0 = sb + warp * SPW + sub; j0 < se; j0 += STRIDE * kCombBatch) {
    Triple4 t[kCombBatch];
#pragma unroll
    for (int u = 0; u < kCombBatch; ++u) {
      const int s = min(j0 + u * STRIDE, se - 1);
      t[u].m = __ldg(mrow + s);
      t[u].l = __ldg(lrow + s);
      t[u].o = __ldg(orow + static_cast<size_t>(s) * (D / 4));
    }
#pragma unroll
    for (int u = 0; u < kCombBatch; ++u)
      t[u].m = (j0 + u * STRIDE < se) ? t[u].m * kLog2e : -INFINITY;
#pragma unroll
    for (int w = 1; w < kCombBatch; w <<= 1)
#pragma unroll
      for (int u = 0; u + w < kCombBatch; u += 2 * w) t[u] = lse_merge4(t[u], t[u + w]);
    acc = lse_merge4(acc, t[0]);
  }
  if constexpr (SPW == 2) {
    Triple4 other;
    other.m = __shfl_xor_sync(0xffffffffu, acc.m, LPS);
    other.l = __shfl_xor_sync(0xffffffffu, acc.l, LPS);
    other.o.x = __shfl_xor_sync(0xffffffffu, acc.o.x, LPS);
    other.o.y = __shfl_xor_sync(0xffffffffu, acc.o.y, LPS);
    other.o.z = __shfl_xor_sync(0xffffffffu, acc.o.z, LPS);
    other.o.w = __shfl_xor_sync(0xffffffffu, acc.o.w, LPS);
    acc = sub ? lse_merge4(other, acc) : lse_merge4(acc, other);
  }
  if (sub == 0) red[warp][c4] = acc;
  __syncthreads();
  if (threadIdx.x < LPS) {  // the four warp triples, pairwise in two levels
    const Triple4 a = lse_merge4(red[0][threadIdx.x], red[1][threadIdx.x]);
    const Triple4 b = lse_merge4(red[2][threadIdx.x], red[3][threadIdx.x]);
    const Triple4 r = lse_merge4(a, b);
    const size_t si = static_cast<size_t>(row) * nseg + seg;
    reinterpret_cast<float4*>(o2 + si * D)[threadIdx.x] = r.o;
    if (threadIdx.x == 0) {
      m2[si] = (r.m == -INFINITY) ? -INFINITY : r.m * kLn2;
      l2[si] = r.l;
    }
  }
}

// grid.x = rows * C with clusters of C CTAs along x: CTA (row, segment).
template <int D, int NW>
__global__ void __launch_bounds__(NW * 32)
    lse_combine_kernel(const float* __restrict__ pm, const float* __restrict__ pl,
                       const float* __restrict__ po, void* out, float* lse, int S, int o_f32) {
  constexpr int LPS = D / 4;     // lanes per partial (four columns each)
  constexpr int SPW = 32 / LPS;  // partials per warp load
  __shared__ Triple4 red[NW][LPS];
  __shared__ Triple4 cta_res[LPS];
  grid_dependency_wait();  // the partials of a preceding decode grid are complete
  const uint32_t rank = cluster_ctarank();
  const uint32_t csize = cluster_nctarank();
  const long long row = blockIdx.x / csize;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane / LPS, c4 = lane % LPS;
  const int per = (S + static_cast<int>(csize) - 1) / static_cast<int>(csize);
  const int sb = static_cast<int>(rank) * per, se = min(S, sb + per);
  const float* mrow = pm + row * S;
  const float* lrow = pl + row * S;
  const float4* orow = reinterpret_cast<const float4*>(po + row * S * D) + c4;

  Triple4 acc{-INFINITY, 0.f, make_float4(0.f, 0.f, 0.f, 0.f)};
  constexpr int STRIDE = NW * SPW;
  for (int j0 = sb + warp * SPW + sub; j0 < se; j0 += STRIDE * kCombBatch) {
    Triple4 t[kCombBatch];
    // All 3 x 8 loads are issued before any is used: no branch around them
    // (an index past the segment is clamped, and its triple masked to the
    // identity afterwards), so they are all in flight together.
#pragma unroll
    for (int u = 0; u < kCombBatch; ++u) {
      const int s = min(j0 + u * STRIDE, se - 1);
      t[u].m = __ldg(mrow + s);
      t[u].l = __ldg(lrow + s);
      t[u].o = __ldg(orow + static_cast<size_t>(s) * (D / 4));
    }
#pragma unroll
    for (int u = 0; u < kCombBatch; ++u)  // -inf stays -inf: an empty split, its o never used
      t[u].m = (j0 + u * STRIDE < se) ? t[u].m * kLog2e : -INFINITY;
#pragma unroll
    for (int w = 1; w < kCombBatch; w <<= 1)
#pragma unroll
      for (int u = 0; u + w < kCombBatch; u += 2 * w) t[u] = lse_merge4(t[u], t[u + w]);
    acc = lse_merge4(acc, t[0]);
  }
  if constexpr (SPW == 2) {  // the two partials of a warp load share columns
    Triple4 other;
    other.m = __shfl_xor_sync(0xffffffffu, acc.m, LPS);
    other.l = __shfl_xor_sync(0xffffffffu, acc.l, LPS);
    other.o.x = __shfl_xor_sync(0xffffffffu, acc.o.x, LPS);
    other.o.y = __shfl_xor_sync(0xffffffffu, acc.o.y, LPS);
    other.o.z = __shfl_xor_sync(0xffffffffu, acc.o.z, LPS);
    other.o.w = __shfl_xor_sync(0xffffffffu, acc.o.w, LPS);
    acc = sub ? lse_merge4(other, acc) : lse_merge4(acc, other);
  }
  if (sub == 0) red[warp][c4] = acc;
  __syncthreads();
#pragma unroll
  for (int w = NW / 2; w >= 1; w >>= 1) {  // warp triples, pairwise in log2(NW) levels
    if (warp < w && sub == 0) red[warp][c4] = lse_merge4(red[warp][c4], red[warp + w][c4]);
    __syncthreads();
  }
  if (threadIdx.x < LPS) cta_res[threadIdx.x] = red[0][threadIdx.x];
  cluster_sync_all();  // every CTA's triple is in its shared memory
  if (rank == 0 && threadIdx.x < LPS) {
    Triple4 t[kCombMaxCluster];
#pragma unroll
    for (int r = 0; r < kCombMaxCluster; ++r) {
      t[r].m = -INFINITY;
      if (r < static_cast<int>(csize)) {
        const uint32_t a = dsmem_map(&cta_res[threadIdx.x], static_cast<uint32_t>(r));
        t[r].m = ld_dsmem_f32(a + offsetof(Triple4, m));
        t[r].l = ld_dsmem_f32(a + offsetof(Triple4, l));
        t[r].o = ld_dsmem_f32x4(a + offsetof(Triple4, o));
      }
    }
#pragma unroll
    for (int w = 1; w < kCombMaxCluster; w <<= 1)
#pragma unroll
      for (int u = 0; u + w < kCombMaxCluster; u += 2 * w) t[u] = lse_merge4(t[u], t[u + w]);
    const Triple4 r = t[0];
    const float inv = (r.l > 0.f) ? 1.f / r.l : 0.f;
    const float4 v = make_float4(r.o.x * inv, r.o.y * inv, r.o.z * inv, r.o.w * inv);
    const size_t oi = static_cast<size_t>(row) * D + 4 * threadIdx.x;
    if (o_f32) {
      *reinterpret_cast<float4*>(static_cast<float*>(out) + oi) = v;
    } else {
      uint2 w;
      w.x = pack_bf16x2(v.x, v.y);
      w.y = pack_bf16x2(v.z, v.w);
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + oi) = w;
    }
    if (threadIdx.x == 0) lse[row] = (r.l > 0.f) ? (r.m + __log2f(r.l)) * kLn2 : -INFINITY;
  }
  cluster_sync_all();  // CTA 0 has read the others' shared memory before they exit
}

}  // namespace b300
