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
// Persistent CTAs, one per SM: each CTA walks a list of work items (a 256-row
// query block of one (batch, head)), so that the loads and MMAs of the next
// item overlap the epilogue of the current one.  Items are dealt to the CTAs
// in a zig-zag over a heaviest-first order (causal), which balances the
// triangular work without any global counter.
//
// CTA layout (384 threads):
//   warp 0      TMA producer: Q tiles of each item, then K_j, V_j into a STAGES-deep ring
//   warp 1      MMA issuer (whole warp, one elected lane): S_i = Q_i K_j^T, O_i += P_i V_j
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
//
// Barriers (all waits bounded in time):
//   q_full / q_empty         Q tile i of an item landed / its last S MMA done (per Q buffer)
//   kv_full[s] / kv_empty[s] ring stage s landed / its MMAs done
//   s_full[i]                S_i of the current key tile is in tensor memory
//   p_full[i]                P_i written (and O_i rescaled) by the 128 softmax threads
//   o_full[i] / o_empty[i]   O_i of an item complete / read out by the epilogue
#pragma once

#include "ptx.cuh"

namespace b300 {

__device__ unsigned int g_prefill_status;  // OR of kStatus* bits (bounded waits that ran out)

constexpr unsigned kStatusProducer = 1u, kStatusMma = 2u, kStatusSoftmax = 4u;
// A paged prefill met a block-table entry outside [0, num_pages): the keys of
// that page were read as zeros (an input error, not a timeout).
constexpr unsigned kStatusPrefillBadPage = 4096u;

// Maximum number of sequences of one variable-length launch (the per-CTA item
// table lives in shared memory).
constexpr int kMaxVarlenSeqs = 4096;
// P_i(j) V_j is issued in this many parts along the keys (32-key chunks
// grouped evenly).  The softmax signals each part as soon as its columns of
// P are written, so the tensor core starts O += P V on the first keys while
// the exponentials of the last keys are still being computed.  Two parts pay
// in FP8, whose tensor work per tile is half of bf16's while its softmax is
// not shorter (2-3 % faster measured); in bf16 they measured no faster than
// one.
__host__ __device__ constexpr int pv_parts(bool fp8) { return fp8 ? 2 : 1; }
constexpr int kPvPartsMax = 2;

// Two layouts share one kernel.  Dense: B sequences of N tokens,
// q [B, N, Hq, d], LSE [B, Hq, N].  Variable length: `cu_seqlens[0..num_seqs]`
// (int32, device) holds the first token of each sequence in packed
// q [T, Hq, d], k/v [T, Hkv, d] (T = total_rows), LSE [Hq, T].  Either way the
// tensor maps see a [rows, heads, d] array and every item carries its
// sequence's first row and length.
struct PrefillParams {
  void* o;
  float* lse;
  const int* cu_seqlens;  // NULL: dense layout
  int B, Hq, Hkv, N;      // dense: batch and sequence length
  int num_seqs, total_rows;
  int causal, window, o_f32;
  int nqb;           // dense: number of 256-row query blocks per sequence
  int n_items;       // dense: nqb * B * Hq (variable length: counted on the device)
  float scale_log2;  // scale * log2(e): scores are kept in base-2 units
  // FP8 (dense layout only): a stored code c stands for c * 2^-e, with e the
  // exponent of its 128-row tile (Q, K) or of its head (V)
  const int* q_exp;  // [B, Hq, nt]
  const int* k_exp;  // [B, Hkv, nt]
  const int* v_exp;  // [B, Hkv]
  int nt;            // 128-row tiles per sequence
  // Paged K/V (dense layout of q): K, V are [num_pages, page_size, Hkv, d] and
  // key j of sequence b is row j % page_size of page
  // block_table[b * pages_per_seq + j / page_size]; page_size is a multiple
  // of 64, the rows of one TMA box.
  const int* block_table;
  int page_size, pages_per_seq, num_pages;
};

template <int D, bool FP8 = false>
struct PrefillCfg {
  static constexpr int EB = FP8 ? 1 : 2;  // bytes per element of Q, K, V
  static constexpr int BM = 128;  // query rows per Q tile (one softmax warpgroup)
  static constexpr int BN = 128;  // keys per K/V tile
  static constexpr int DCH = D * EB / 128;  // 128-byte swizzle atoms across d
  static constexpr int TILE_BYTES = BM * D * EB;  // one Q, K or V tile
  // Q is double-buffered (the next item's Q loads while the current item
  // runs) when shared memory allows: at d=64 and in FP8 always; at d=128 in
  // bf16 the K/V ring would have to shrink to three stages, so one Q buffer
  // is kept there.
  static constexpr int QBUF = (D == 128 && !FP8) ? 1 : 2;
  static constexpr int STAGES = FP8 ? 8 : ((D == 128) ? 4 : 8);
  static constexpr int RING_OFF = QBUF * 2 * TILE_BYTES;
  static constexpr int BAR_OFF = RING_OFF + STAGES * TILE_BYTES;
  // + barriers and the TMEM address (512 B), the variable-length item table
  // (kMaxVarlenSeqs + 1 ints), alignment slack
  static constexpr int TABLE_OFF = BAR_OFF + 512;
  static constexpr int SMEM_BYTES = TABLE_OFF + (kMaxVarlenSeqs + 1) * 4 + 1024;
  static constexpr int THREADS = 384;
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(BM == BN, "Q and K/V tiles share one byte layout");
};

// The k-th work item of CTA c among G CTAs: zig-zag over the item order.
__device__ __forceinline__ int prefill_item(int c, int k, int G) {
  return (k & 1) ? k * G + (G - 1 - c) : k * G + c;
}

// What one work item covers: query block qb of head h of sequence b (whose
// tokens are rows [base, base + n) of the [rows, heads, d] view), and the
// key-tile range [jlo[i], jhi[i]] of each of its two Q tiles.
struct PrefillItem {
  int qb, b, h, hk;
  int base, n;
  int jlo[2], jhi[2];
  bool act[2];
  int J0, J1;
};

// First row and length of variable-length sequence s, clamped so that every
// row the kernel touches lies inside [0, total_rows) whatever cu_seqlens holds.
__device__ __forceinline__ void varlen_seq(const PrefillParams& p, int s, int& base, int& n) {
  B300_DCHECK(p.cu_seqlens[s] >= 0 && p.cu_seqlens[s] <= p.cu_seqlens[s + 1] &&
                  p.cu_seqlens[s + 1] <= p.total_rows,
              kDbgCuSeqlens);
  const int a = min(max(p.cu_seqlens[s], 0), p.total_rows);
  const int e = min(max(p.cu_seqlens[s + 1], a), p.total_rows);
  base = a;
  n = e - a;
}

// `table[s]` (s = 0..num_seqs) is the number of items of sequences 0..s-1
// (variable-length layout only).
template <bool VARLEN>
__device__ __forceinline__ PrefillItem prefill_item_info(const PrefillParams& p, int item,
                                                         const int* table) {
  constexpr int BN = 128;
  PrefillItem it;
  if constexpr (VARLEN) {
    int lo = 0, hi = p.num_seqs - 1;  // last s with table[s] <= item
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (table[mid] <= item) lo = mid; else hi = mid - 1;
    }
    it.b = lo;
    varlen_seq(p, lo, it.base, it.n);
    const int nqb = (it.n + 255) / 256;
    const int local = item - table[lo];
    if (p.causal) {  // heaviest query blocks of the sequence first
      it.qb = nqb - 1 - local / p.Hq;
      it.h = local % p.Hq;
    } else {
      it.qb = local % nqb;
      it.h = local / nqb;
    }
  } else {
    const int BH = p.B * p.Hq;
    int bh;
    if (p.causal) {  // heaviest query blocks first
      it.qb = p.nqb - 1 - item / BH;
      bh = item % BH;
    } else {  // all blocks of one head together: they share its K/V in L2
      it.qb = item % p.nqb;
      bh = item / p.nqb;
    }
    it.b = bh / p.Hq;
    it.h = bh % p.Hq;
    it.base = it.b * p.N;
    it.n = p.N;
  }
  it.hk = it.h / (p.Hq / p.Hkv);
  const int N = it.n;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r0 = it.qb * 256 + i * 128;
    it.act[i] = r0 < N;
    const int r1 = min(r0 + 127, N - 1);
    const int klo = (p.window >= 0) ? max(0, r0 - p.window) : 0;
    const int khi = p.causal ? r1 : ((p.window >= 0) ? min(N - 1, r1 + p.window) : N - 1);
    it.jlo[i] = klo / BN;
    it.jhi[i] = khi / BN;
  }
  it.J0 = it.act[1] ? min(it.jlo[0], it.jlo[1]) : it.jlo[0];
  it.J1 = it.act[1] ? max(it.jhi[0], it.jhi[1]) : it.jhi[0];
  B300_DCHECK(it.b >= 0 && it.b < p.num_seqs && it.h >= 0 && it.h < p.Hq && it.qb >= 0 &&
                  (!it.act[0] || (it.jlo[0] <= it.jhi[0] && it.jhi[0] * BN < it.n)) &&
                  (!it.act[1] || (it.jlo[1] <= it.jhi[1] && it.jhi[1] * BN < it.n)),
              kDbgPrefillItem);
  return it;
}

// VARLEN selects the layout at compile time, so that the dense launch carries
// none of the variable-length bookkeeping.
//
// FP8 selects e4m3 operands (dense layout, d = 128): Q and K tiles as in bf16
// but one byte per element, V stored transposed ([B, Hkv, d, Np], so that the
// PV product reads it K-major), tcgen05 kind::f8f6f4 with 32 elements of K
// per instruction.  The softmax multiplies the raw scores by
// scale * 2^-(e_Q + e_K) of the tile pair, writes P rounded to e4m3 into
// tensor memory over the first 32 columns of its S (four keys to a column,
// the A operand of PV), and the epilogue divides by l and by 2^e_V.  The lazy
// rescale keeps P <= 2^8 < 448, inside e4m3.
//
// PAGED selects K and V gathered from a page pool through a block table
// (dense layout of q, bf16): each 128-key tile is two 64-row TMA boxes, each
// from the page that holds its keys.
template <int D, bool VARLEN, bool FP8 = false, bool PAGED = false>
__global__ void __launch_bounds__(384, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
  static_assert(!FP8 || (D == 128 && !VARLEN), "FP8: dense layout, d = 128");
  static_assert(!PAGED || (!FP8 && !VARLEN), "paged K/V: dense bf16 layout");
  using C = PrefillCfg<D, FP8>;
  constexpr int BN = C::BN;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sRing = smem + C::RING_OFF;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* q_full = bars;                   // [QBUF][2]
  uint64_t* q_empty = q_full + 2 * C::QBUF;  // [QBUF][2]
  uint64_t* kv_full = q_empty + 2 * C::QBUF; // [STAGES]
  uint64_t* kv_empty = kv_full + STAGES;  // [STAGES]
  uint64_t* s_full = kv_empty + STAGES;   // [2]
  uint64_t* p_full = s_full + 2;          // [2]
  uint64_t* o_full = p_full + 2;          // [2]
  uint64_t* o_empty = o_full + 2;         // [2]
  uint64_t* mma_done = o_empty + 2;
  constexpr int kPvParts = pv_parts(FP8);
  static_assert(kPvParts >= 1 && kPvParts <= kPvPartsMax && 4 % kPvParts == 0,
                "parts of the four 32-key chunks");
  uint64_t* p_part = mma_done + 1;  // [2][kPvParts - 1]: leading parts of P_i written
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(p_part + 2 * (kPvPartsMax - 1));
  int* table = reinterpret_cast<int*>(smem + C::TABLE_OFF);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = gridDim.x;
  const int c = blockIdx.x;

  // Variable length: items per sequence (query blocks x heads), prefix-summed
  // into the shared table by a block-wide scan.
  int n_items = p.n_items;
  if constexpr (VARLEN) {
    constexpr int PER = (kMaxVarlenSeqs + C::THREADS - 1) / C::THREADS;
    int cnt[PER];
    int mine = 0;
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int s = threadIdx.x * PER + u;
      cnt[u] = 0;
      if (s < p.num_seqs) {
        int b0, n0;
        varlen_seq(p, s, b0, n0);
        cnt[u] = (n0 + 255) / 256 * p.Hq;
      }
      mine += cnt[u];
    }
    int incl = mine;  // inclusive scan over the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    __shared__ int warp_sum[C::THREADS / 32];
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    int before = incl - mine;
    for (int w = 0; w < warp; ++w) before += warp_sum[w];
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int s = threadIdx.x * PER + u;
      if (s <= p.num_seqs) table[s] = before;
      before += cnt[u];
    }
    __syncthreads();
    n_items = table[p.num_seqs];
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2 * C::QBUF; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
      mbar_init(&o_full[i], 1);
      mbar_init(&o_empty[i], 128);
    }
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    mbar_init(mma_done, 1);
    for (int x = 0; x < 2 * (kPvParts - 1); ++x) mbar_init(&p_part[x], 128);
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

  // Register split: launched at 168 per thread (384 x 168 = 64512); warpgroup
  // 0 (producer, MMA issuer, allocator, idle) gives back to 136 and the two softmax
  // warpgroups take 184: 128 x 136 + 256 x 184 = 64512.
  if (warp < 4) {
  setmaxnreg_dec<136>();
  if (warp == 0) {
    // ================================================================ producer
    if (lane == 0) {
      bool ok = true;
      int issued = 0;  // K/V ring loads issued so far (all items)
      int k = 0;       // items of this CTA started
      for (int item = prefill_item(c, 0, G); item < n_items && ok;
           item = prefill_item(c, ++k, G)) {
        const PrefillItem it = prefill_item_info<VARLEN>(p, item, table);
        // Q tile i of this item, once the last S MMA of the previous item
        // has read the buffer.
        const int qs = k % C::QBUF, qr = k / C::QBUF;  // Q buffer and its reuse count
        for (int i = 0; i < 2 && ok; ++i) {
          uint64_t* qf = &q_full[qs * 2 + i];
          if (qr > 0 && !(ok = mbar_wait(&q_empty[qs * 2 + i], (qr - 1) & 1, &g_prefill_status,
                                         kStatusProducer)))
            break;
          mbar_arrive_expect_tx(qf, C::TILE_BYTES);
          for (int cc = 0; cc < C::DCH; ++cc)
            tma_load_3d(sQ + (qs * 2 + i) * C::TILE_BYTES + cc * (C::BM * 128), &tm_q, qf,
                        cc * (128 / C::EB), it.h, it.base + it.qb * 256 + i * 128);
        }
        const int nloads = 2 * (it.J1 - it.J0 + 1);  // K_j, V_j alternate in the ring
        for (int u = 0; u < nloads && ok; ++u, ++issued) {
          const int s = issued % STAGES;
          if (issued >= STAGES &&
              !(ok = mbar_wait(&kv_empty[s], ((issued / STAGES) - 1) & 1, &g_prefill_status,
                               kStatusProducer)))
            break;
          mbar_arrive_expect_tx(&kv_full[s], C::TILE_BYTES);
          const int j = it.J0 + u / 2;
          if constexpr (FP8) {
            if (u & 1)  // V^T tile: keys [j*BN, j*BN + BN) x all of d, of plane (b, hk)
              tma_load_3d(sRing + s * C::TILE_BYTES, &tm_v, &kv_full[s], j * BN, 0,
                          it.b * p.Hkv + it.hk);
            else
              tma_load_3d(sRing + s * C::TILE_BYTES, &tm_k, &kv_full[s], 0, it.hk,
                          it.base + j * BN);
          } else if constexpr (PAGED) {
            // two 64-key boxes, each from its own page; keys past the
            // sequence's end use page coordinate num_pages, which TMA fills
            // with zeros (the block table is not read there)
            const CUtensorMap* tm = (u & 1) ? &tm_v : &tm_k;
            for (int hh = 0; hh < 2; ++hh) {
              const int kr = j * BN + hh * 64;
              int page = p.num_pages, prow = 0;
              if (kr < it.n) {
                const int e =
                    p.block_table[static_cast<size_t>(it.b) * p.pages_per_seq + kr / p.page_size];
                if (e >= 0 && e < p.num_pages) {
                  page = e;
                  prow = kr % p.page_size;
                } else {
                  atomicOr(&g_prefill_status, kStatusPrefillBadPage);
                }
              }
              for (int cc = 0; cc < C::DCH; ++cc)
                tma_load_4d(sRing + s * C::TILE_BYTES + cc * (BN * 128) + hh * 64 * 128, tm,
                            &kv_full[s], cc * 64, it.hk, prow, page);
            }
          } else {
            const CUtensorMap* tm = (u & 1) ? &tm_v : &tm_k;
            for (int cc = 0; cc < C::DCH; ++cc)
              tma_load_3d(sRing + s * C::TILE_BYTES + cc * (BN * 128), tm, &kv_full[s], cc * 64,
                          it.hk, it.base + j * BN);
          }
        }
      }
      // Every issued copy has landed before the CTA may exit (a no-op wait on
      // the normal path, where the MMA warp already consumed them all).
      for (int u = max(0, issued - STAGES); u < issued; ++u)
        mbar_wait(&kv_full[u % STAGES], (u / STAGES) & 1, &g_prefill_status, kStatusProducer);
      for (int kk = max(0, k - C::QBUF); kk < k; ++kk)
        for (int i = 0; i < 2; ++i)
          mbar_wait(&q_full[(kk % C::QBUF) * 2 + i], (kk / C::QBUF) & 1, &g_prefill_status,
                    kStatusProducer);
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    // The whole warp runs this loop (waits included); one elected lane issues
    // each tcgen05 instruction.  Descriptors are a base plus constant offsets.
    const uint32_t idS = FP8 ? idesc_e4m3_f32(128, BN) : idesc_bf16_f32(128, BN, false);
    const uint32_t idO = FP8 ? idesc_e4m3_f32(128, D) : idesc_bf16_f32(128, D, true);
    const uint64_t dq0 = smem_desc_sw128(smem_u32(sQ), 16, 1024);
    const uint64_t dk0 = smem_desc_sw128(smem_u32(sRing), 16, 1024);
    const uint64_t dv0 = smem_desc_sw128(smem_u32(sRing), BN * 128, 1024);
    uint32_t pcnt[2] = {0u, 0u};  // p_full phases consumed, per Q tile
    uint32_t ocnt[2] = {0u, 0u};  // items in which Q tile i was active
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, &g_prefill_status, kStatusMma));
    };

    // S_i = Q_i K^T: K-major operands, 32 bytes of d per instruction (16
    // bf16 or 32 e4m3 elements).
    int qs = 0;  // Q buffer of the current item
    auto issue_S = [&](int i, int stage) {
      const uint64_t a0 = dq0 + static_cast<uint64_t>(((qs * 2 + i) * C::TILE_BYTES) >> 4);
      const uint64_t b0 = dk0 + static_cast<uint64_t>((stage * C::TILE_BYTES) >> 4);
#pragma unroll
      for (int kk = 0; kk < D * C::EB / 32; ++kk) {
        const uint32_t off = ((kk >> 2) * (C::BM * 128) + (kk & 3) * 32) >> 4;
        if constexpr (FP8)
          umma_ss_f8_warp(tmem + i * 128, a0 + off, b0 + off, idS, kk > 0 ? 1u : 0u);
        else
          umma_ss_warp(tmem + i * 128, a0 + off, b0 + off, idS, kk > 0 ? 1u : 0u);
      }
      umma_commit_warp(&s_full[i]);
    };
    // O_i += P_i V.  P from tensor memory (bf16 pairs or e4m3 quadruples in
    // the first columns of S_i).  bf16: V MN-major in shared memory, 16 keys
    // per instruction.  FP8: V^T K-major in shared memory, 32 keys per
    // instruction.
    // Part `part` of kPvParts covers keys [part, part + 1) * BN / kPvParts.
    auto issue_PV = [&](int i, int stage, bool accumulate, int part) {
      if constexpr (FP8) {
        constexpr int KK = BN / 32 / kPvParts;
        const uint64_t b0 = dk0 + static_cast<uint64_t>((stage * C::TILE_BYTES) >> 4);
#pragma unroll
        for (int x = 0; x < KK; ++x) {
          const int kk = part * KK + x;
          umma_ts_f8_warp(tmem + 256 + i * D, tmem + i * 128 + kk * 8, b0 + ((kk * 32) >> 4), idO,
                          (accumulate || kk > 0) ? 1u : 0u);
        }
      } else {
        constexpr int KK = BN / 16 / kPvParts;
        const uint64_t b0 = dv0 + static_cast<uint64_t>((stage * C::TILE_BYTES) >> 4);
#pragma unroll
        for (int x = 0; x < KK; ++x) {
          const int kk = part * KK + x;
          umma_ts_warp(tmem + 256 + i * D, tmem + i * 128 + kk * 8, b0 + ((kk * 16 * 128) >> 4),
                       idO, (accumulate || kk > 0) ? 1u : 0u);
        }
      }
    };

    bool ok = true;
    int t0 = 0;  // ring position of this item's first load (K_J0)
    int k = 0;
    for (int item = prefill_item(c, 0, G); item < n_items && ok;
         item = prefill_item(c, ++k, G)) {
      const PrefillItem it = prefill_item_info<VARLEN>(p, item, table);
      qs = k % C::QBUF;
      for (int i = 0; i < 2 && ok; ++i) ok = wait(&q_full[qs * 2 + i], (k / C::QBUF) & 1);
      if (ok) ok = wait(&kv_full[t0 % STAGES], (t0 / STAGES) & 1);
      if (!ok) break;
      tc_fence_after();
      for (int i = 0; i < 2; ++i) {
        if (it.act[i] && it.J0 >= it.jlo[i] && it.J0 <= it.jhi[i]) {
          issue_S(i, t0 % STAGES);
          if (it.jhi[i] == it.J0) umma_commit_warp(&q_empty[qs * 2 + i]);
        } else if (!it.act[i]) {
          umma_commit_warp(&q_empty[qs * 2 + i]);  // no S MMA reads this Q tile
        }
      }
      umma_commit_warp(&kv_empty[t0 % STAGES]);
      int t = t0 + 1;  // ring position of V_j
      for (int j = it.J0; j <= it.J1 && ok; ++j, t += 2) {
        const int sv = t % STAGES;
        if (!(ok = wait(&kv_full[sv], (t / STAGES) & 1))) break;
        tc_fence_after();
        if constexpr (!FP8) {
          // A tile that runs past the sequence's end holds the next
          // sequence's rows (or TMA's zero fill) there.  Their scores are
          // masked, so P = 0 for them, but 0 times a non-finite value is not
          // 0: zero those V rows (whole 128-byte rows of every swizzle
          // chunk) before the tensor core reads the stage.  FP8 needs no
          // fix-up: its transposed V is zero past the sequence's end.
          const int nv = it.n - j * BN;  // >= 1: every visited tile starts inside
          if (nv < BN) {
            uint8_t* vt = sRing + sv * C::TILE_BYTES;
#pragma unroll 1
            for (int cc = 0; cc < C::DCH; ++cc) {
              uint4* z = reinterpret_cast<uint4*>(vt + cc * (BN * 128) + nv * 128);
#pragma unroll 1
              for (int e = lane; e < (BN - nv) * 8; e += 32) z[e] = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();  // generic writes -> tensor-core operand
            __syncwarp();
          }
        }
        const bool has_next = j < it.J1;
        const int sk = (t + 1) % STAGES;
        bool k_ready = false;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          if (!ok) break;
          if (it.act[i] && j >= it.jlo[i] && j <= it.jhi[i]) {
            // each part of P_i once the softmax has written it; the item's
            // first part also once the epilogue has read the previous O_i
#pragma unroll
            for (int part = 0; part < kPvParts && ok; ++part) {
              uint64_t* pb = (part + 1 < kPvParts) ? &p_part[i * (kPvParts - 1) + part] : &p_full[i];
              if (!(ok = wait(pb, pcnt[i] & 1))) break;
              if (part == 0 && j == it.jlo[i] && ocnt[i] > 0 &&
                  !(ok = wait(&o_empty[i], (ocnt[i] - 1) & 1)))
                break;
              tc_fence_after();
              issue_PV(i, sv, j != it.jlo[i], part);
            }
            if (!ok) break;
            ++pcnt[i];
            if (j == it.jhi[i]) {
              umma_commit_warp(&o_full[i]);
              ++ocnt[i];
            }
          }
          if (has_next && it.act[i] && j + 1 >= it.jlo[i] && j + 1 <= it.jhi[i]) {
            if (!k_ready) {
              if (!(ok = wait(&kv_full[sk], ((t + 1) / STAGES) & 1))) break;
              tc_fence_after();
              k_ready = true;
            }
            issue_S(i, sk);
            if (j + 1 == it.jhi[i]) umma_commit_warp(&q_empty[qs * 2 + i]);
          }
        }
        if (!ok) break;
        umma_commit_warp(&kv_empty[sv]);
        if (has_next) {
          if (!k_ready && !(ok = wait(&kv_full[sk], ((t + 1) / STAGES) & 1))) break;
          umma_commit_warp(&kv_empty[sk]);
        }
      }
      t0 += 2 * (it.J1 - it.J0 + 1);
    }
    // All MMAs of this CTA complete before tensor memory is released.
    umma_commit_warp(mma_done);
    wait(mma_done, 0);
  }
  } else {
    setmaxnreg_inc<184>();
    // ================================================================ softmax
    const int i = (warp - 4) >> 2;   // Q tile of this warpgroup
    const int quarter = warp & 3;    // tensor-memory lane quarter this warp may access
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_off + i * 128;
    const uint32_t tO = tmem + lane_off + 256 + i * D;
    const float sl2 = p.scale_log2;
    const bool causal = p.causal != 0;
    const int window = p.window;
    bool ok = true;
    uint32_t scnt = 0;  // s_full phases consumed
    uint32_t ocnt = 0;  // items in which this Q tile was active
    int k = 0;
    for (int item = prefill_item(c, 0, G); item < n_items && ok;
         item = prefill_item(c, ++k, G)) {
      const PrefillItem it = prefill_item_info<VARLEN>(p, item, table);
      const bool act = i ? it.act[1] : it.act[0];  // selects: no run-time index into `it`
      const int jlo = i ? it.jlo[1] : it.jlo[0];
      const int jhi = i ? it.jhi[1] : it.jhi[0];
      if (!act) continue;
      const int r0 = it.qb * 256 + i * 128;
      const int row = r0 + r;
      float m_ref = -INFINITY;  // base-2 running maximum actually used for P
      float l = 0.f;
      // FP8: per-tile score multiplier scale * log2(e) * 2^-(e_Q + e_K); the
      // exponent of the next key tile is loaded one tile ahead
      const int* kexp = nullptr;
      float qsc = 1.f;
      int ek_next = 0;
      if constexpr (FP8) {
        qsc = pow2i(-p.q_exp[(static_cast<size_t>(it.b) * p.Hq + it.h) * p.nt + it.qb * 2 + i]);
        kexp = p.k_exp + (static_cast<size_t>(it.b) * p.Hkv + it.hk) * p.nt;
        ek_next = kexp[jlo];
      }
      for (int j = jlo; j <= jhi; ++j, ++scnt) {
        float c = sl2;
        if constexpr (FP8) {
          c = fmaxf(sl2 * qsc * pow2i(-ek_next), 1e-30f);
          if (j < jhi) ek_next = kexp[j + 1];
        }
        ok = mbar_wait(&s_full[i], scnt & 1, &g_prefill_status, kStatusSoftmax);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        // S row of this thread: four 32-column loads in flight, one wait
        uint32_t u[4][32];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tmem_ld32(tS + cc * 32, u[cc]);
        tmem_wait_ld();
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) reg_fence(u[cc]);
        float s[128];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
#pragma unroll
          for (int e = 0; e < 32; ++e) s[cc * 32 + e] = __uint_as_float(u[cc][e]);
        const int kv0 = j * BN;
        const bool need_mask =
            (kv0 + BN > it.n) || (causal && kv0 + BN - 1 > r0) ||
            (window >= 0 && (r0 + 127 - kv0 > window || (!causal && kv0 + BN - 1 - r0 > window)));
        // Mask: columns [lo_c, hi_c] of this tile are visible to this row.
        // Each 32-column chunk that is visible in every row of the warp is
        // skipped; the others get a per-column select.  One code path serves
        // masked and unmasked tiles (the kernel's instructions must stay
        // within the instruction cache).
        if (need_mask) {
          int lo = 0, hi = it.n - 1;
          if (causal) hi = min(hi, row);
          if (window >= 0) {
            lo = max(lo, row - window);
            if (!causal) hi = min(hi, row + window);
          }
          const int lo_c = lo - kv0, hi_c = hi - kv0;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (__all_sync(0xffffffffu, lo_c <= 32 * q && hi_c >= 32 * q + 31)) continue;
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int cc = 32 * q + e;
              s[cc] = (cc >= lo_c && cc <= hi_c) ? s[cc] : -INFINITY;
            }
          }
        }
        // row maximum: four independent chains of three-input max
        float mc[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int cc = 0; cc < 128; cc += 8)
#pragma unroll
          for (int t = 0; t < 4; ++t) mc[t] = fmax3(mc[t], s[cc + 2 * t], s[cc + 2 * t + 1]);
        const float mx = fmaxf(fmax3(mc[0], mc[1], mc[2]), mc[3]);
        const float m_new = fmaxf(m_ref, mx * c);
        const bool resc = m_new > m_ref + kRescaleThreshold;
        float alpha = 1.f;
        if (resc) {
          alpha = ex2_approx(m_ref - m_new);  // 0 when m_ref = -inf
          m_ref = m_new;
          l *= alpha;
        }
        const float neg_mu = (m_ref == -INFINITY) ? 0.f : -m_ref;
        // Rescale this row of O (only rows whose maximum moved; the previous
        // P V of this tile is complete because S_i(j) was committed after
        // it).  It runs before the first part of P is released, after which
        // the tensor core may add into O, and after that part's exponentials,
        // whose scores no longer need registers.
        auto rescale_o = [&]() {
          if (j > jlo && __any_sync(0xffffffffu, resc)) {
#pragma unroll 1
            for (int cc = 0; cc < D / 32; ++cc) {
              uint32_t w[32];
              tmem_ld32_wait(tO + cc * 32, w);
#pragma unroll
              for (int e = 0; e < 32; ++e) w[e] = __float_as_uint(__uint_as_float(w[e]) * alpha);
              tmem_st32(tO + cc * 32, w);
            }
          }
        };
        // P = 2^(s*scale*log2e - m) on column pairs (packed f32x2 FMA), row sum
        // in four packed partial sums; bf16 pairs or e4m3 quadruples into the
        // first columns of S in tensor memory
        const float2 sl2x2 = make_float2(c, c);
        const float2 nmu2 = make_float2(neg_mu, neg_mu);
        float2 lacc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                          make_float2(0.f, 0.f)};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t pk[16];
          float pv[32];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 x =
                ffma2(make_float2(s[q * 32 + 2 * e], s[q * 32 + 2 * e + 1]), sl2x2, nmu2);
            const float2 pe = make_float2(ex2_approx(x.x), ex2_approx(x.y));
            lacc[e & 3] = fadd2(lacc[e & 3], pe);
            if constexpr (FP8) {
              pv[2 * e] = pe.x;
              pv[2 * e + 1] = pe.y;
            } else {
              pk[e] = pack_bf16x2(pe.x, pe.y);
            }
          }
          if constexpr (FP8) {
            // keys 32q .. 32q+31: columns 8q .. 8q+7, four keys to a column
            uint32_t p8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              p8[e] = pack_e4m3x4(pv[4 * e], pv[4 * e + 1], pv[4 * e + 2], pv[4 * e + 3]);
            tmem_st8(tS + q * 8, p8);
          } else {
            tmem_st16(tS + q * 16, pk);
          }
          // a leading part of P is complete: the tensor core may start on it
          constexpr int QP = 4 / kPvParts;  // 32-key chunks per part
          if ((q + 1) % QP == 0 && q + 1 < 4) {
            if (q + 1 == QP) rescale_o();
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&p_part[i * (kPvParts - 1) + (q + 1) / QP - 1]);
          }
        }
        if constexpr (kPvParts == 1) rescale_o();
        {
          const float2 a = fadd2(lacc[0], lacc[1]), b2 = fadd2(lacc[2], lacc[3]);
          const float2 t = fadd2(a, b2);
          l += t.x + t.y;
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&p_full[i]);
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      ok = mbar_wait(&o_full[i], ocnt & 1, &g_prefill_status, kStatusSoftmax);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ++ocnt;
      tc_fence_after();
      uint32_t u[D / 32][32];
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) tmem_ld32(tO + cc * 32, u[cc]);
      tmem_wait_ld();
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) reg_fence(u[cc]);
      // O_i is in registers: the next item's first P V may overwrite it.
      tc_fence_before();
      mbar_arrive(&o_empty[i]);
      float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      if constexpr (FP8) inv_l *= pow2i(-p.v_exp[static_cast<size_t>(it.b) * p.Hkv + it.hk]);
      if (row < it.n) {
        const size_t orow = (static_cast<size_t>(it.base) + row) * p.Hq + it.h;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          if (p.o_f32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + orow * D + cc * 32);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              dst[e] = make_float4(__uint_as_float(u[cc][4 * e]) * inv_l,
                                   __uint_as_float(u[cc][4 * e + 1]) * inv_l,
                                   __uint_as_float(u[cc][4 * e + 2]) * inv_l,
                                   __uint_as_float(u[cc][4 * e + 3]) * inv_l);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + orow * D +
                                                  cc * 32);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              uint4 w;
              w.x = pack_bf16x2(__uint_as_float(u[cc][8 * e + 0]) * inv_l,
                                __uint_as_float(u[cc][8 * e + 1]) * inv_l);
              w.y = pack_bf16x2(__uint_as_float(u[cc][8 * e + 2]) * inv_l,
                                __uint_as_float(u[cc][8 * e + 3]) * inv_l);
              w.z = pack_bf16x2(__uint_as_float(u[cc][8 * e + 4]) * inv_l,
                                __uint_as_float(u[cc][8 * e + 5]) * inv_l);
              w.w = pack_bf16x2(__uint_as_float(u[cc][8 * e + 6]) * inv_l,
                                __uint_as_float(u[cc][8 * e + 7]) * inv_l);
              dst[e] = w;
            }
          }
        }
        const size_t li = VARLEN
                              ? static_cast<size_t>(it.h) * p.total_rows + it.base + row
                              : (static_cast<size_t>(it.b) * p.Hq + it.h) * it.n + row;
        p.lse[li] =
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
