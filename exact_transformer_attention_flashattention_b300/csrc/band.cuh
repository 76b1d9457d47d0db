// Prefill for a short non-causal sliding window (the local attention of the
// Arabic thread on extending context length, point 1: tokens attend only to
// their neighbours), d = 64, dense layout.  Same method as prefill_kernel
// (tiles of Q, K, V on chip, online softmax, exact normalisation: "FlashAttention"
// learn page, "Technical insight"), scheduled for short key ranges.
//
// A 128-row Q tile of a band of width w sees only ceil((2w + 128) / 128) + 1
// key tiles (three for w = 128).  With so few key tiles per Q tile, pairing two
// Q tiles in one work item (as prefill_kernel does) leaves the tensor core and
// one softmax warpgroup idle at every item boundary.  Here each softmax
// warpgroup owns an independent stream of Q tiles with its own K/V ring, Q
// buffers, and S, P, O in tensor memory:
//
//   warps 0, 2  TMA producers of streams 0 and 1 (warp 2 first allocates
//               tensor memory)
//   warps 1, 3  MMA issuers of streams 0 and 1
//   warps 4-7   softmax + epilogue of stream 0
//   warps 8-11  softmax + epilogue of stream 1
//
// A stream is a sequence of steps (Q tile n, key tile j); step g's K and V sit
// at positions 2g and 2g + 1 of the stream's ring.  The MMA warp issues
// S(g+1) as soon as the softmax has read S(g) into registers -- across Q tile
// boundaries too -- so a softmax pass never waits for its S, and P(g) V(g)
// goes in as soon as P(g) is written.  The two streams share only the tensor
// core, the MUFU units and the memory system: each has its own warps, so a
// wait in one never delays the other.
//
// Tensor memory, stream s at columns [256 s, 256 s + 256):
//   S [0,128)   P [128,192) (bf16 pairs)   O [192, 192 + D)
#pragma once

#include "prefill.cuh"

namespace b300 {

// bits of g_prefill_status
constexpr unsigned kStatusBandProducer = 8192u, kStatusBandMma = 16384u,
                   kStatusBandSoftmax = 32768u;

template <int D>
struct BandCfg {
  static constexpr int BM = 128, BN = 128;
  static constexpr int DCH = D * 2 / 128;          // 128-byte swizzle atoms across d
  static constexpr int TILE_BYTES = BM * D * 2;    // one Q, K or V tile
  static constexpr int RS = 4;                     // K/V ring stages per stream
  static constexpr int QB = 2;                     // Q buffers per stream
  static constexpr int RING_OFF = 2 * QB * TILE_BYTES;
  static constexpr int OST_OFF = RING_OFF + 2 * RS * TILE_BYTES;  // O staging, one tile per stream
  static constexpr int BAR_OFF = OST_OFF + 2 * TILE_BYTES;
  static constexpr int BARS_PER_STREAM = 20;
  static constexpr int SMEM_BYTES = BAR_OFF + 512 + 1024;  // + barriers, TMEM address, alignment
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
  static constexpr int THREADS = 384;
  static constexpr int TM_S = 0, TM_P = 128, TM_O = 192, TM_STREAM = 256;
  static_assert(D == 64, "the band schedule is built for d = 64");
  static_assert(TM_O + D <= TM_STREAM, "one stream's tensor-memory columns");
};

// Q tile x of the launch (x over B * Hq * nt, (batch, head)-major; the host
// keeps B * Hq * nt below 2^31) and the key tiles [jlo, jhi] its rows can see.
struct BandTile {
  int b, h, hk, r0, jlo, jhi;
};

__device__ __forceinline__ BandTile band_tile(const PrefillParams& p, int x, int nt) {
  BandTile t;
  const int bh = x / nt;
  t.r0 = (x - bh * nt) * 128;
  t.b = bh / p.Hq;
  t.h = bh - t.b * p.Hq;
  t.hk = t.h / (p.Hq / p.Hkv);
  const int r1 = min(t.r0 + 127, p.N - 1);
  t.jlo = max(0, t.r0 - p.window) / 128;
  t.jhi = min(p.N - 1, r1 + p.window) / 128;
  B300_DCHECK(t.b < p.B && t.r0 < p.N && t.jlo <= t.jhi, kDbgBandTile);
  return t;
}

template <int D>
__global__ void __launch_bounds__(384, 1)
    prefill_band_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_o, const PrefillParams p) {
  using C = BandCfg<D>;
  constexpr int BN = C::BN, RS = C::RS, QB = C::QB;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;                  // [stream][QB] tiles
  uint8_t* sRing = smem + C::RING_OFF; // [stream][RS] tiles
  uint8_t* sOst = smem + C::OST_OFF;   // [stream] O tile, 128-byte swizzled rows
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  // per stream s, at bars + 20 s:
  auto q_full = [&](int s, int b) { return bars + s * C::BARS_PER_STREAM + b; };
  auto q_empty = [&](int s, int b) { return bars + s * C::BARS_PER_STREAM + 2 + b; };
  auto kv_full = [&](int s, int st) { return bars + s * C::BARS_PER_STREAM + 4 + st; };
  auto kv_empty = [&](int s, int st) { return bars + s * C::BARS_PER_STREAM + 8 + st; };
  auto s_full = [&](int s) { return bars + s * C::BARS_PER_STREAM + 12; };
  auto s_free = [&](int s) { return bars + s * C::BARS_PER_STREAM + 13; };
  auto p_full = [&](int s) { return bars + s * C::BARS_PER_STREAM + 14; };
  auto pv_done = [&](int s) { return bars + s * C::BARS_PER_STREAM + 15; };
  auto o_full = [&](int s) { return bars + s * C::BARS_PER_STREAM + 16; };
  auto o_empty = [&](int s) { return bars + s * C::BARS_PER_STREAM + 17; };
  auto st_full = [&](int s) { return bars + s * C::BARS_PER_STREAM + 18; };
  auto st_free = [&](int s) { return bars + s * C::BARS_PER_STREAM + 19; };
  uint64_t* mma_done = bars + 2 * C::BARS_PER_STREAM;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 2);  // mma_done: one per stream

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // this CTA's Q tiles: a contiguous run of the (batch, head)-major order;
  // stream s takes every other one, from offset s
  const int nt = (p.N + 127) / 128;
  const long long T = static_cast<long long>(p.B) * p.Hq * nt;
  const int lo = static_cast<int>(T * blockIdx.x / gridDim.x);
  const int hi = static_cast<int>(T * (blockIdx.x + 1) / gridDim.x);
  auto n_tiles = [&](int s) -> int { return hi - lo > s ? (hi - lo - s + 1) / 2 : 0; };
  auto tile_of = [&](int s, int n) { return band_tile(p, lo + s + 2 * n, nt); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      for (int b = 0; b < QB; ++b) {
        mbar_init(q_full(s, b), 1);
        mbar_init(q_empty(s, b), 1);
      }
      for (int st = 0; st < RS; ++st) {
        mbar_init(kv_full(s, st), 1);
        mbar_init(kv_empty(s, st), 1);
      }
      mbar_init(s_full(s), 1);
      mbar_init(s_free(s), 128);
      mbar_init(p_full(s), 128);
      mbar_init(pv_done(s), 1);
      mbar_init(o_full(s), 1);
      mbar_init(o_empty(s), 128);
      mbar_init(st_full(s), 128);
      mbar_init(st_free(s), 1);
    }
    mbar_init(mma_done, 1);
    mbar_init(mma_done + 1, 1);
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    if (!p.o_f32) tma_prefetch_desc(&tm_o);
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Register split: 128 x 104 + 256 x 200 = 384 x 168 (the launch total); the
  // softmax warps hold a 128-column row of S in registers.
  if (warp < 4) {
    setmaxnreg_dec<104>();
    const int s = warp >> 1;  // stream served by this warp
    const int ns = n_tiles(s);
    if ((warp & 1) == 0) {
      // ======================================= producer of stream s (warps 0, 2)
      if (lane == 0) {
        int pos = 0, nq = 0;  // K/V loads and Q loads issued
        bool ok = true;
        for (int n = 0; n < ns && ok; ++n) {
          const BandTile t = tile_of(s, n);
          const int qb = n % QB;
          if (n >= QB)
            ok = mbar_wait(q_empty(s, qb), ((n / QB) - 1) & 1, &g_prefill_status,
                           kStatusBandProducer);
          if (!ok) break;
          mbar_arrive_expect_tx(q_full(s, qb), C::TILE_BYTES);
          for (int cc = 0; cc < C::DCH; ++cc)
            tma_load_3d(sQ + (s * QB + qb) * C::TILE_BYTES + cc * (C::BM * 128), &tm_q,
                        q_full(s, qb), cc * 64, t.h, t.b * p.N + t.r0);
          ++nq;
          for (int j = t.jlo; j <= t.jhi && ok; ++j)
            for (int kv = 0; kv < 2; ++kv, ++pos) {
              const int st = pos % RS;
              if (pos >= RS &&
                  !(ok = mbar_wait(kv_empty(s, st), ((pos / RS) - 1) & 1, &g_prefill_status,
                                   kStatusBandProducer)))
                break;
              mbar_arrive_expect_tx(kv_full(s, st), C::TILE_BYTES);
              for (int cc = 0; cc < C::DCH; ++cc)
                tma_load_3d(sRing + (s * RS + st) * C::TILE_BYTES + cc * (BN * 128),
                            kv ? &tm_v : &tm_k, kv_full(s, st), cc * 64, t.hk,
                            t.b * p.N + j * BN);
            }
        }
        // every issued copy has landed before the CTA may exit
        for (int u = max(0, pos - RS); u < pos; ++u)
          mbar_wait(kv_full(s, u % RS), (u / RS) & 1, &g_prefill_status, kStatusBandProducer);
        for (int u = max(0, nq - QB); u < nq; ++u)
          mbar_wait(q_full(s, u % QB), (u / QB) & 1, &g_prefill_status, kStatusBandProducer);
      }
    } else {
      // ========================================= MMA issuer of stream s (warps 1, 3)
      // Order: S(0), S(1), P(0)V(0), S(2), P(1)V(1), ...: S(g+1) needs only the
      // softmax's read of S(g), which comes before its P(g).
      const uint32_t idS = idesc_bf16_f32(128, BN, false);
      const uint32_t idO = idesc_bf16_f32(128, D, true);
      const uint64_t dq0 = smem_desc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dk0 = smem_desc_sw128(smem_u32(sRing), 16, 1024);
      const uint64_t dv0 = smem_desc_sw128(smem_u32(sRing), BN * 128, 1024);
      const uint32_t tS = tmem + s * C::TM_STREAM + C::TM_S;
      const uint32_t tP = tmem + s * C::TM_STREAM + C::TM_P;
      const uint32_t tO = tmem + s * C::TM_STREAM + C::TM_O;
      auto wait = [&](uint64_t* bar, uint32_t parity) {
        return __all_sync(0xffffffffu,
                          mbar_wait(bar, parity, &g_prefill_status, kStatusBandMma));
      };
      // P(g) V(g) for key tile j of tile n (first / last key tile of that tile)
      auto pv = [&](int g, int n, int j, bool first, bool last) -> bool {
        const int vp = 2 * g + 1;
        if (!wait(p_full(s), g & 1) || !wait(kv_full(s, vp % RS), (vp / RS) & 1)) return false;
        if (first && n > 0 && !wait(o_empty(s), (n - 1) & 1)) return false;
        tc_fence_after();
        uint8_t* vt = sRing + (s * RS + vp % RS) * C::TILE_BYTES;
        // V rows past the sequence's end hold the next sequence's rows: their
        // P is 0, but 0 times a non-finite value is not; zero them
        const int nv = p.N - j * BN;
        if (nv < BN) {
#pragma unroll 1
          for (int cc = 0; cc < C::DCH; ++cc) {
            uint4* z = reinterpret_cast<uint4*>(vt + cc * (BN * 128) + nv * 128);
#pragma unroll 1
            for (int e = lane; e < (BN - nv) * 8; e += 32) z[e] = make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        const uint64_t b0 = dv0 + static_cast<uint64_t>((smem_u32(vt) - smem_u32(sRing)) >> 4);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          umma_ts_warp(tO, tP + kk * 8, b0 + ((kk * 16 * 128) >> 4), idO,
                       (!first || kk > 0) ? 1u : 0u);
        umma_commit_warp(pv_done(s));
        umma_commit_warp(kv_empty(s, vp % RS));
        if (last) umma_commit_warp(o_full(s));
        return true;
      };
      bool ok = true;
      int g = 0;
      // the step whose P V is still to be issued
      int pn = -1, pj = 0;
      bool pfirst = false, plast = false;
      for (int n = 0; n < ns && ok; ++n) {
        const BandTile t = tile_of(s, n);
        const int qb = n % QB;
        for (int j = t.jlo; j <= t.jhi; ++j, ++g) {
          const int kp = 2 * g;
          ok = (g == 0 || wait(s_free(s), (g - 1) & 1)) &&
               (j != t.jlo || wait(q_full(s, qb), (n / QB) & 1)) &&
               wait(kv_full(s, kp % RS), (kp / RS) & 1);
          if (!ok) break;
          tc_fence_after();
          const uint64_t a0 = dq0 + static_cast<uint64_t>(((s * QB + qb) * C::TILE_BYTES) >> 4);
          const uint64_t b0 =
              dk0 + static_cast<uint64_t>(((s * RS + kp % RS) * C::TILE_BYTES) >> 4);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * (C::BM * 128) + (kk & 3) * 32) >> 4;
            umma_ss_warp(tS, a0 + off, b0 + off, idS, kk > 0 ? 1u : 0u);
          }
          umma_commit_warp(s_full(s));
          umma_commit_warp(kv_empty(s, kp % RS));
          if (j == t.jhi) umma_commit_warp(q_empty(s, qb));
          if (pn >= 0 && !(ok = pv(g - 1, pn, pj, pfirst, plast))) break;
          pn = n;
          pj = j;
          pfirst = j == t.jlo;
          plast = j == t.jhi;
        }
      }
      if (ok && pn >= 0) pv(g - 1, pn, pj, pfirst, plast);
      // All MMAs of this warp complete before tensor memory is released.
      umma_commit_warp(mma_done + s);
      wait(mma_done + s, 0);
    }
  } else {
    setmaxnreg_inc<200>();
    // ================================================================ softmax
    const int s = (warp - 4) >> 2;  // stream of this warpgroup
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_off + s * C::TM_STREAM + C::TM_S;
    const uint32_t tP = tmem + lane_off + s * C::TM_STREAM + C::TM_P;
    const uint32_t tO = tmem + lane_off + s * C::TM_STREAM + C::TM_O;
    const bool issuer = quarter == 0 && lane == 0;  // issues this stream's O stores
    uint8_t* ost = sOst + s * C::TILE_BYTES;
    const float c = p.scale_log2;
    const int window = p.window;
    const int ns = n_tiles(s);
    bool ok = true;

    // Epilogue of tile e (its tile, final base-2 maximum and row sum): O from
    // tensor memory, normalised by 1/l, to the output; LSE from m and l.  It
    // runs after the next tile's first step, whose wait for P V of the step
    // before also covers this tile's last P V.
    auto epilogue = [&](int e, const BandTile& t, float m_fin, float l_fin) -> bool {
      if (!__all_sync(0xffffffffu,
                      mbar_wait(o_full(s), e & 1, &g_prefill_status, kStatusBandSoftmax)))
        return false;
      tc_fence_after();
      const float inv_l = (l_fin > 0.f) ? 1.f / l_fin : 0.f;
      const int row = t.r0 + r;
      uint32_t pk[D / 2];  // bf16 pairs of this row of O / l
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t w[32];
        tmem_ld32(tO + cc * 32, w);
        tmem_wait_ld();
        reg_fence(w);
        if (p.o_f32) {
          if (row < p.N) {
            float4* dst = reinterpret_cast<float4*>(
                static_cast<float*>(p.o) +
                ((static_cast<size_t>(t.b) * p.N + row) * p.Hq + t.h) * D + cc * 32);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              dst[q] = make_float4(__uint_as_float(w[4 * q]) * inv_l,
                                   __uint_as_float(w[4 * q + 1]) * inv_l,
                                   __uint_as_float(w[4 * q + 2]) * inv_l,
                                   __uint_as_float(w[4 * q + 3]) * inv_l);
          }
        } else {
#pragma unroll
          for (int q = 0; q < 16; ++q)
            pk[cc * 16 + q] = pack_bf16x2(__uint_as_float(w[2 * q]) * inv_l,
                                          __uint_as_float(w[2 * q + 1]) * inv_l);
        }
      }
      tc_fence_before();
      mbar_arrive(o_empty(s));  // the next tile's first P V may overwrite O
      if (!p.o_f32) {
        // bf16 O: the tile goes through shared memory and one TMA store (rows
        // past the sequence's end fall outside the map and are not written).
        // The previous tile's store must have finished reading the staging
        // buffer first.
        if (e > 0) {
          if (issuer) {
            bulk_wait_group_read0();
            mbar_arrive(st_free(s));
          }
          if (!__all_sync(0xffffffffu, mbar_wait(st_free(s), (e - 1) & 1, &g_prefill_status,
                                                 kStatusBandSoftmax)))
            return false;
        }
        // row r of the staging tile: 16-byte chunk k at (k ^ (r % 8)) * 16
        uint8_t* orow = ost + r * 128;
#pragma unroll
        for (int k = 0; k < 8; ++k)
          *reinterpret_cast<uint4*>(orow + ((k ^ (r & 7)) << 4)) =
              make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
        fence_proxy_async_smem();
        mbar_arrive(st_full(s));
        if (issuer) {
          if (!mbar_wait(st_full(s), e & 1, &g_prefill_status, kStatusBandSoftmax)) return false;
          tma_store_4d(&tm_o, ost, 0, t.h, t.r0, t.b);
          bulk_commit_group();
        }
      }
      if (row < p.N)
        p.lse[(static_cast<size_t>(t.b) * p.Hq + t.h) * p.N + row] =
            (l_fin > 0.f) ? (m_fin + __log2f(l_fin)) * kLn2 : -INFINITY;
      return true;
    };

    uint32_t g = 0;  // stream steps done
    BandTile prev{};
    float m_prev = -INFINITY, l_prev = 0.f;
    for (int n = 0; n < ns && ok; ++n) {
      const BandTile t = tile_of(s, n);
      const int row = t.r0 + r;
      float m_ref = -INFINITY;  // base-2 running maximum actually used for P
      float l = 0.f;
      for (int j = t.jlo; j <= t.jhi; ++j, ++g) {
        ok = __all_sync(0xffffffffu,
                        mbar_wait(s_full(s), g & 1, &g_prefill_status, kStatusBandSoftmax));
        if (!ok) break;
        tc_fence_after();
        uint32_t u[4][32];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tmem_ld32(tS + cc * 32, u[cc]);
        tmem_wait_ld();
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) reg_fence(u[cc]);
        tc_fence_before();
        mbar_arrive(s_free(s));  // S may now be overwritten by the next S MMA
        float x[128];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
#pragma unroll
          for (int e = 0; e < 32; ++e) x[cc * 32 + e] = __uint_as_float(u[cc][e]);
        const int kv0 = j * BN;
        // Visible columns of this row: [lo_c, hi_c].  Each 32-column chunk is,
        // for the warp as a whole, fully visible, empty (no exponentials: P = 0)
        // or mixed (a per-lane visibility mask selects -inf).
        uint32_t empty = 0;  // bit q: chunk q is masked for every row of the warp
        if (kv0 + BN > p.N || t.r0 + 127 - kv0 > window || kv0 + BN - 1 - t.r0 > window) {
          const int lo_c = max(0, row - window) - kv0;
          const int hi_c = min(p.N - 1, row + window) - kv0;
          // the warp's extreme bounds decide each chunk's class uniformly
          const int lo_min = __reduce_min_sync(0xffffffffu, lo_c);
          const int lo_max = __reduce_max_sync(0xffffffffu, lo_c);
          const int hi_min = __reduce_min_sync(0xffffffffu, hi_c);
          const int hi_max = __reduce_max_sync(0xffffffffu, hi_c);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (lo_max <= 32 * q && hi_min >= 32 * q + 31) continue;
            if (lo_min > 32 * q + 31 || hi_max < 32 * q) {
              empty |= 1u << q;
              continue;
            }
            const int a = lo_c - 32 * q, b = hi_c - 32 * q;  // visible: a <= e <= b
            const uint32_t hi_bits = b >= 31 ? 0xffffffffu : (b < 0 ? 0u : (2u << b) - 1u);
            const uint32_t lo_bits = a <= 0 ? 0xffffffffu : (a > 31 ? 0u : ~((1u << a) - 1u));
            const uint32_t vis = hi_bits & lo_bits;
#pragma unroll
            for (int e = 0; e < 32; ++e)
              x[32 * q + e] = (vis & (1u << e)) ? x[32 * q + e] : -INFINITY;
          }
        }
        // row maximum: eight independent chains, then empty chunks dropped (their
        // scores were not masked)
        float mc[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)  // chain k: chunk k / 2, column pairs 2 (k % 2) + 4 i
          mc[k] = fmaxf(x[32 * (k >> 1) + 2 * (k & 1)], x[32 * (k >> 1) + 2 * (k & 1) + 1]);
#pragma unroll
        for (int e = 4; e < 32; e += 4)
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mc[k] = fmax3(mc[k], x[32 * (k >> 1) + e + 2 * (k & 1)],
                          x[32 * (k >> 1) + e + 2 * (k & 1) + 1]);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          mc[2 * q] = (empty & (1u << q)) ? -INFINITY : fmaxf(mc[2 * q], mc[2 * q + 1]);
        const float mx = fmaxf(fmaxf(mc[0], mc[2]), fmaxf(mc[4], mc[6]));
        const float m_new = fmaxf(m_ref, mx * c);
        const bool resc = m_new > m_ref + kRescaleThreshold;
        float alpha = 1.f;
        if (resc) {
          alpha = ex2_approx(m_ref - m_new);  // 0 when m_ref = -inf
          m_ref = m_new;
          l *= alpha;
        }
        const float neg_mu = (m_ref == -INFINITY) ? 0.f : -m_ref;
        // P(g-1) V is done before P is rewritten or O rescaled
        if (g > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(pv_done(s), (g - 1) & 1, &g_prefill_status,
                                                 kStatusBandSoftmax));
          if (!ok) break;
        }
        tc_fence_after();
        const float2 c2 = make_float2(c, c);
        const float2 nmu2 = make_float2(neg_mu, neg_mu);
        float2 lacc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                          make_float2(0.f, 0.f)};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t pk[16];
          if (empty & (1u << q)) {
#pragma unroll
            for (int e = 0; e < 16; ++e) pk[e] = 0u;
            tmem_st16(tP + q * 16, pk);
            continue;
          }
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 y = ffma2(make_float2(x[q * 32 + 2 * e], x[q * 32 + 2 * e + 1]), c2, nmu2);
            const float2 pe = make_float2(ex2_approx(y.x), ex2_approx(y.y));
            lacc[e & 3] = fadd2(lacc[e & 3], pe);
            pk[e] = pack_bf16x2(pe.x, pe.y);
          }
          tmem_st16(tP + q * 16, pk);
        }
        {
          const float2 a = fadd2(lacc[0], lacc[1]), b2 = fadd2(lacc[2], lacc[3]);
          const float2 sum = fadd2(a, b2);
          l += sum.x + sum.y;
        }
        if (j > t.jlo && __any_sync(0xffffffffu, resc)) {
#pragma unroll 1
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t w[32];
            tmem_ld32_wait(tO + cc * 32, w);
#pragma unroll
            for (int e = 0; e < 32; ++e) w[e] = __float_as_uint(__uint_as_float(w[e]) * alpha);
            tmem_st32(tO + cc * 32, w);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(p_full(s));
        // the previous tile's epilogue, now that its last P V is done
        if (j == t.jlo && n > 0 && !(ok = epilogue(n - 1, prev, m_prev, l_prev))) break;
      }
      prev = t;
      m_prev = m_ref;
      l_prev = l;
    }
    if (ok && ns > 0) epilogue(ns - 1, prev, m_prev, l_prev);
    // every O store of this stream has completed before the CTA exits
    if (issuer && !p.o_f32) bulk_wait_group0();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace b300
