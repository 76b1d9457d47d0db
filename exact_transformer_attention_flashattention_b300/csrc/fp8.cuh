// FP8 (e4m3) quantisation of the attention inputs: bf16 Q, K, V in, e4m3
// codes plus one power-of-two exponent per tile out.
//
// FlashAttention-3 computes attention in FP8 ("FlashAttention" learn page,
// aiunderstanding.org, section on the future of FlashAttention; FlashAttention-3
// article, ybx.com, "FlashAttention-3 innovations" item 3).  The scaling used
// here: a tile shares the largest integer e with amax * 2^e <= 448, and each
// value x is stored as e4m3(x * 2^e), rounded to nearest even.  Q and K are
// tiled by 128 rows of one (batch, head); V has one exponent per (batch,
// head) and is stored transposed, [B, Hkv, d, Np] with the key axis padded to
// Np = N rounded up to 16, so that both tensor-core products read K-major
// operands.
//
// Two launches: fp8_vamax_kernel writes the absolute maximum of every
// 128-key tile of V; fp8_quantize_kernel then runs one CTA per 128-row tile of
// Q, of K and of V (V reduces its head's tile maxima first).  A quantisation
// CTA brings its tile into shared memory with one bulk copy per row, so its
// bytes are in flight without holding registers and more CTAs fit on an SM.
#pragma once

#include "prefill.cuh"  // g_prefill_status, which also reports this file's bounded wait
#include "ptx.cuh"

namespace b300 {

// bit of g_prefill_status: the quantisation kernel gave up waiting for its tile
constexpr unsigned kStatusFp8Stage = 1u << 20;

// Untiled bulk copy global -> shared of `bytes` (a multiple of 16, both
// addresses 16-byte aligned), completion signalled on `bar` (tx bytes).
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

struct Fp8QuantParams {
  const __nv_bfloat16* q;  // [B, N, Hq, D]
  const __nv_bfloat16* k;  // [B, N, Hkv, D]
  const __nv_bfloat16* v;  // [B, N, Hkv, D]
  uint8_t* q8;             // [B, N, Hq, D]
  uint8_t* k8;             // [B, N, Hkv, D]
  uint8_t* v8t;            // [B, Hkv, D, Np]
  int* q_exp;              // [B, Hq, nt]
  int* k_exp;              // [B, Hkv, nt]
  int* v_exp;              // [B, Hkv]
  float* v_tile_amax;      // [B, Hkv, nt] (workspace)
  int B, Hq, Hkv, N, Np, nt;
};

constexpr int kFp8QuantThreads = 256;

// Largest e with amax * 2^e <= 448, clamped to [-126, 126]; 0 for an all-zero
// tile.  amax = 1.f * 2^(be-127) with be its biased exponent: 448 = 1.75 * 2^8,
// so e = 8 - (be - 127) when the significand is at most 1.75, one less above.
__device__ __forceinline__ int fp8_scale_exponent(float amax) {
  if (!(amax > 0.f)) return 0;
  const uint32_t b = __float_as_uint(amax);
  const int be = static_cast<int>((b >> 23) & 0xFFu);
  if (be == 0) return 126;  // subnormal maximum: the clamp
  const int e = 135 - be - (((b & 0x7FFFFFu) > 0x600000u) ? 1 : 0);
  return min(max(e, -126), 126);
}

__device__ __forceinline__ float absmax8(const uint4& w, float m) {
  m = fmaxf(m, fmaxf(fabsf(bf16lo_to_f32(w.x)), fabsf(bf16hi_to_f32(w.x))));
  m = fmaxf(m, fmaxf(fabsf(bf16lo_to_f32(w.y)), fabsf(bf16hi_to_f32(w.y))));
  m = fmaxf(m, fmaxf(fabsf(bf16lo_to_f32(w.z)), fabsf(bf16hi_to_f32(w.z))));
  m = fmaxf(m, fmaxf(fabsf(bf16lo_to_f32(w.w)), fabsf(bf16hi_to_f32(w.w))));
  return m;
}

// Maximum over the CTA (256 threads); every thread gets the result.
__device__ __forceinline__ float block_max256(float m, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = m;
  __syncthreads();
  m = red[0];
#pragma unroll
  for (int w = 1; w < kFp8QuantThreads / 32; ++w) m = fmaxf(m, red[w]);
  return m;
}

// Tile t of one (b, h) of a [B, N, H, D] bf16 tensor: rows t*128 .. t*128+127
// (those below N).  Thread mapping of the row-major loads: pass u covers rows
// u*16 + tid/16, 8 elements of d at (tid % 16) * 8.
template <int D>
__device__ __forceinline__ const uint4* tile_row_ptr(const __nv_bfloat16* x, int b, int h, int H,
                                                     int N, int row) {
  return reinterpret_cast<const uint4*>(x + ((static_cast<size_t>(b) * N + row) * H + h) * D);
}

template <int D>
__global__ void __launch_bounds__(kFp8QuantThreads)
    fp8_vamax_kernel(const Fp8QuantParams p) {
  static_assert(D == 128, "one 16-byte load per thread and row covers 8 of d");
  __shared__ float red[kFp8QuantThreads / 32];
  const int t = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x;
  float m = 0.f;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int row = t * 128 + u * 16 + tid / 16;
    if (row < p.N) m = absmax8(tile_row_ptr<D>(p.v, b, hk, p.Hkv, p.N, row)[tid % 16], m);
  }
  m = block_max256(m, red);
  if (tid == 0) p.v_tile_amax[(static_cast<size_t>(b) * p.Hkv + hk) * p.nt + t] = m;
}

template <int D>
__global__ void __launch_bounds__(kFp8QuantThreads)
    fp8_quantize_kernel(const Fp8QuantParams p) {
  static_assert(D == 128, "tile mappings assume d = 128");
  __shared__ float red[kFp8QuantThreads / 32];
  // the tile's rows (row r at r * 2D bytes); a V tile's transpose, [d][128
  // keys] of e4m3, reuses its first 16 KB once the rows are in registers
  __shared__ __align__(128) uint8_t sX[128 * D * 2];
  __shared__ uint64_t xbar;
  uint8_t* sT = sX;
  const int tid = threadIdx.x;
  // Rows t*128 .. of head h of x into sX: one 2D-byte bulk copy per row
  // inside the sequence; false if the copies did not land in time.
  auto stage = [&](const __nv_bfloat16* x, int b, int h, int H, int t) -> bool {
    const int nrows = min(128, p.N - t * 128);
    if (tid == 0) {
      mbar_init(&xbar, 1);
      fence_mbar_init();
      mbar_arrive_expect_tx(&xbar, static_cast<uint32_t>(nrows) * D * 2);
    }
    __syncthreads();
    if (tid < nrows)
      bulk_load(sX + tid * D * 2, tile_row_ptr<D>(x, b, h, H, p.N, t * 128 + tid), D * 2, &xbar);
    return mbar_wait(&xbar, 0, &g_prefill_status, kStatusFp8Stage);
  };
  const long long nq = static_cast<long long>(p.B) * p.Hq * p.nt;
  const long long nk = static_cast<long long>(p.B) * p.Hkv * p.nt;
  long long job = blockIdx.x;

  if (job < nq + nk) {
    // ------------------------------------------------------------- Q or K tile
    const bool isq = job < nq;
    if (!isq) job -= nq;
    const int H = isq ? p.Hq : p.Hkv;
    const __nv_bfloat16* x = isq ? p.q : p.k;
    uint8_t* y = isq ? p.q8 : p.k8;
    int* ex = isq ? p.q_exp : p.k_exp;
    const int t = static_cast<int>(job % p.nt);
    const int h = static_cast<int>((job / p.nt) % H);
    const int b = static_cast<int>(job / (static_cast<long long>(p.nt) * H));
    if (tid == 0) B300_DCHECK(b < p.B, kDbgFp8Job);
    stage(x, b, h, H, t);
    // the rows are read twice from shared memory, for the maximum and for
    // the codes, so that no register holds them across the reduction
    float m = 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int rr = u * 16 + tid / 16;  // row within the tile
      if (t * 128 + rr < p.N) m = absmax8(reinterpret_cast<const uint4*>(sX + rr * D * 2)[tid % 16], m);
    }
    m = block_max256(m, red);
    const int e = fp8_scale_exponent(m);
    const float s = pow2i(e);
    if (tid == 0) ex[(static_cast<size_t>(b) * H + h) * p.nt + t] = e;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int rr = u * 16 + tid / 16;
      const int row = t * 128 + rr;
      if (row >= p.N) continue;
      const uint4 w = reinterpret_cast<const uint4*>(sX + rr * D * 2)[tid % 16];
      uint2 o;
      o.x = pack_e4m3x4(bf16lo_to_f32(w.x) * s, bf16hi_to_f32(w.x) * s,
                        bf16lo_to_f32(w.y) * s, bf16hi_to_f32(w.y) * s);
      o.y = pack_e4m3x4(bf16lo_to_f32(w.z) * s, bf16hi_to_f32(w.z) * s,
                        bf16lo_to_f32(w.w) * s, bf16hi_to_f32(w.w) * s);
      reinterpret_cast<uint2*>(y + ((static_cast<size_t>(b) * p.N + row) * H + h) * D)[tid % 16] = o;
    }
    return;
  }

  // ----------------------------------------------------------------- V tile
  job -= nq + nk;
  const int t = static_cast<int>(job % p.nt);
  const int hk = static_cast<int>((job / p.nt) % p.Hkv);
  const int b = static_cast<int>(job / (static_cast<long long>(p.nt) * p.Hkv));
  if (tid == 0) B300_DCHECK(b < p.B, kDbgFp8Job);
  const size_t bh = static_cast<size_t>(b) * p.Hkv + hk;
  // Transposing mapping: lane = group of 4 consecutive keys (4*lane .. 4*lane+3),
  // warp w covers 8 elements of d at w*8 and w*8 + 64.  Each thread packs the
  // 4 keys of one d into a 32-bit word of the transposed tile.  The tile's
  // loads are issued before the head's maximum is reduced, so both are in
  // flight together.
  const int rg = tid & 31, cg = tid >> 5;
  float m = 0.f;
  for (int u = tid; u < p.nt; u += kFp8QuantThreads) m = fmaxf(m, p.v_tile_amax[bh * p.nt + u]);
  stage(p.v, b, hk, p.Hkv, t);
  m = block_max256(m, red);
  const int e = fp8_scale_exponent(m);
  const float s = pow2i(e);
  if (tid == 0 && t == 0) p.v_exp[bh] = e;
  uint4 wt[2][4];
#pragma unroll
  for (int pass = 0; pass < 2; ++pass)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int rr = 4 * rg + i;  // row within the tile
      wt[pass][i] = make_uint4(0u, 0u, 0u, 0u);
      if (t * 128 + rr < p.N) wt[pass][i] = reinterpret_cast<const uint4*>(sX + rr * D * 2)[cg + 8 * pass];
    }
  __syncthreads();  // every row read before the transpose overwrites them
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    const int c8 = cg + 8 * pass;  // 16-byte column of d
    const uint4* w = wt[pass];
    float f[4][8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[i][0] = bf16lo_to_f32(w[i].x); f[i][1] = bf16hi_to_f32(w[i].x);
      f[i][2] = bf16lo_to_f32(w[i].y); f[i][3] = bf16hi_to_f32(w[i].y);
      f[i][4] = bf16lo_to_f32(w[i].z); f[i][5] = bf16hi_to_f32(w[i].z);
      f[i][6] = bf16lo_to_f32(w[i].w); f[i][7] = bf16hi_to_f32(w[i].w);
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint32_t word = pack_e4m3x4(f[0][c] * s, f[1][c] * s, f[2][c] * s, f[3][c] * s);
      *reinterpret_cast<uint32_t*>(&sT[(c8 * 8 + c) * 128 + 4 * rg]) = word;
    }
  }
  __syncthreads();
  // rows of V^T: 16-byte chunks, eight per d, written while inside [0, Np)
  uint8_t* dst = p.v8t + bh * D * static_cast<size_t>(p.Np) + static_cast<size_t>(t) * 128;
#pragma unroll
  for (int pass = 0; pass < (D * 8) / kFp8QuantThreads; ++pass) {
    const int id = tid + pass * kFp8QuantThreads;
    const int c = id >> 3, kc = id & 7;
    if (t * 128 + kc * 16 < p.Np)
      *reinterpret_cast<uint4*>(dst + static_cast<size_t>(c) * p.Np + kc * 16) =
          *reinterpret_cast<const uint4*>(&sT[c * 128 + kc * 16]);
  }
}

}  // namespace b300
