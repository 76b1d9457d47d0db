// C ABI of the b300attn library: argument validation, TMA tensor-map encoding,
// launch configuration.  All kernels live in this translation unit so that
// their status words can be read back by attn_device_status.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <set>
#include <utility>
#include <string>

#include "b300attn.h"
#include "backward.cuh"
#include "band.cuh"
#include "decode.cuh"
#include "fp8.cuh"
#include "prefill.cuh"

using namespace b300;

namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(B300ATTN_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 4-D bf16 tensor map over a row-major [d3][d2][d1][d0] array (d0 contiguous).
int make_map_4d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                uint64_t d3, uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3,
                CUtensorMapSwizzle swizzle, const char* name) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return fail(B300ATTN_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  const cuuint64_t dims[4] = {d0, d1, d2, d3};
  const cuuint64_t strides[3] = {d0 * 2, d0 * d1 * 2, d0 * d1 * d2 * 2};
  const cuuint32_t box[4] = {b0, b1, b2, b3};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(B300ATTN_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with CUresult %d", name,
                static_cast<int>(r));
  return B300ATTN_OK;
}

// 3-D tensor map over a row-major [d2][d1][d0] array (d0 contiguous) of bf16
// elements, or of bytes when `bytes` is set (e4m3 codes).  `promo` is the L2
// fetch granule: 256 B by default; 128 B for 128-byte rows whose neighbours
// (the next head's row) are read by another CTA much later.
int make_map_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                uint32_t b0, uint32_t b1, uint32_t b2, CUtensorMapSwizzle swizzle,
                const char* name, bool bytes = false,
                CUtensorMapL2promotion promo = CU_TENSOR_MAP_L2_PROMOTION_L2_256B) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return fail(B300ATTN_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  const uint64_t es = bytes ? 1 : 2;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * es, d0 * d1 * es};
  const cuuint32_t box[3] = {b0, b1, b2};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                        3, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                        promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(B300ATTN_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with CUresult %d", name,
                static_cast<int>(r));
  return B300ATTN_OK;
}

// Raises a kernel's dynamic shared-memory limit, once per (kernel, device).
template <typename K>
int set_smem(K kernel, int bytes) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  const auto key = std::make_pair(reinterpret_cast<const void*>(kernel), dev);
  std::lock_guard<std::mutex> lock(mu);
  if (done.count(key)) return B300ATTN_OK;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
  done.insert(key);
  return B300ATTN_OK;
}

// Number of SMs of the current device (cached per device).
int sm_count(int* out) {
  constexpr int kMaxDev = 64;
  static int cache[kMaxDev] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev >= 0 && dev < kMaxDev && cache[dev] > 0) {
    *out = cache[dev];
    return B300ATTN_OK;
  }
  int n = 0;
  e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(MultiProcessorCount)");
  if (n < 1) return fail(B300ATTN_ERR_CUDA, "device reports %d SMs", n);
  if (dev >= 0 && dev < kMaxDev) cache[dev] = n;
  *out = n;
  return B300ATTN_OK;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// `max_items` bounds the number of work items (exact for the dense layout).
template <int D>
int launch_prefill(const void* q, const void* k, const void* v, const PrefillParams& p,
                   long long max_items, cudaStream_t stream) {
  using C = PrefillCfg<D>;
  CUtensorMap tq, tk, tv;
  int rc;
  // q, k, v seen as [rows, heads, d]; tiles of 128 rows x 64 elements of d.
  // At d = 64 a row is 128 B: fetch it alone, not with the next head's row.
  const CUtensorMapL2promotion promo =
      D == 64 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
  if ((rc = make_map_3d(&tq, q, D, p.Hq, p.total_rows, 64, 1, C::BM,
                        CU_TENSOR_MAP_SWIZZLE_128B, "q", false, promo)) != B300ATTN_OK)
    return rc;
  if ((rc = make_map_3d(&tk, k, D, p.Hkv, p.total_rows, 64, 1, C::BN,
                        CU_TENSOR_MAP_SWIZZLE_128B, "k", false, promo)) != B300ATTN_OK)
    return rc;
  if ((rc = make_map_3d(&tv, v, D, p.Hkv, p.total_rows, 64, 1, C::BN,
                        CU_TENSOR_MAP_SWIZZLE_128B, "v", false, promo)) != B300ATTN_OK)
    return rc;
  auto kernel = p.cu_seqlens ? prefill_kernel<D, true> : prefill_kernel<D, false>;
  if ((rc = set_smem(kernel, C::SMEM_BYTES)) != B300ATTN_OK) return rc;
  int sms = 0;
  if ((rc = sm_count(&sms)) != B300ATTN_OK) return rc;
  // persistent: one CTA per SM (the kernel's shared memory admits no second one)
  const int grid = static_cast<int>(std::min<long long>(max_items, sms));
  kernel<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(tq, tk, tv, p);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
  return B300ATTN_OK;
}

// Widest window (keys on each side) that the band schedule takes: a Q tile
// then sees at most five key tiles.
constexpr int kBandMaxWindow = 256;

// Short non-causal window at d = 64, dense layout: the two-stream band kernel.
// A bf16 O is written by TMA through a 4-D map [B][N][Hq][64], so that a
// tile's rows past N are clipped at its own sequence's end.
int launch_prefill_band(const void* q, const void* k, const void* v, const PrefillParams& p,
                        cudaStream_t stream) {
  using C = BandCfg<64>;
  CUtensorMap tq, tk, tv, to;
  int rc;
  // rows are 128 B (d = 64): fetch them alone, not with the next head's row
  const CUtensorMapL2promotion promo = CU_TENSOR_MAP_L2_PROMOTION_L2_128B;
  if ((rc = make_map_3d(&tq, q, 64, p.Hq, p.total_rows, 64, 1, C::BM,
                        CU_TENSOR_MAP_SWIZZLE_128B, "q", false, promo)) != B300ATTN_OK)
    return rc;
  if ((rc = make_map_3d(&tk, k, 64, p.Hkv, p.total_rows, 64, 1, C::BN,
                        CU_TENSOR_MAP_SWIZZLE_128B, "k", false, promo)) != B300ATTN_OK)
    return rc;
  if ((rc = make_map_3d(&tv, v, 64, p.Hkv, p.total_rows, 64, 1, C::BN,
                        CU_TENSOR_MAP_SWIZZLE_128B, "v", false, promo)) != B300ATTN_OK)
    return rc;
  if (p.o_f32)
    to = tq;  // not read: an f32 O is written with plain stores
  else if ((rc = make_map_4d(&to, p.o, 64, p.Hq, p.N, p.B, 64, 1, C::BM, 1,
                             CU_TENSOR_MAP_SWIZZLE_128B, "o")) != B300ATTN_OK)
    return rc;
  if ((rc = set_smem(prefill_band_kernel<64>, C::SMEM_BYTES)) != B300ATTN_OK) return rc;
  int sms = 0;
  if ((rc = sm_count(&sms)) != B300ATTN_OK) return rc;
  const long long tiles = static_cast<long long>(p.B) * p.Hq * ((p.N + 127) / 128);
  const int grid = static_cast<int>(std::min<long long>((tiles + 1) / 2, sms));
  prefill_band_kernel<64><<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(tq, tk, tv, to, p);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "band prefill launch");
  return B300ATTN_OK;
}

// Paged prefill: q dense [B*N, Hq, D] (3-D map, 128-row boxes); K and V
// pools [num_pages, page_size, Hkv, D] (4-D maps, 64-row boxes).
template <int D>
int launch_prefill_paged(const void* q, const void* k_pages, const void* v_pages,
                         const PrefillParams& p, cudaStream_t stream) {
  using C = PrefillCfg<D>;
  CUtensorMap tq, tk, tv;
  int rc;
  if ((rc = make_map_3d(&tq, q, D, p.Hq, p.total_rows, 64, 1, C::BM,
                        CU_TENSOR_MAP_SWIZZLE_128B, "q")) != B300ATTN_OK)
    return rc;
  if ((rc = make_map_4d(&tk, k_pages, D, p.Hkv, p.page_size, p.num_pages, 64, 1, 64, 1,
                        CU_TENSOR_MAP_SWIZZLE_128B, "k_pages")) != B300ATTN_OK)
    return rc;
  if ((rc = make_map_4d(&tv, v_pages, D, p.Hkv, p.page_size, p.num_pages, 64, 1, 64, 1,
                        CU_TENSOR_MAP_SWIZZLE_128B, "v_pages")) != B300ATTN_OK)
    return rc;
  auto kernel = prefill_kernel<D, false, false, true>;
  if ((rc = set_smem(kernel, C::SMEM_BYTES)) != B300ATTN_OK) return rc;
  int sms = 0;
  if ((rc = sm_count(&sms)) != B300ATTN_OK) return rc;
  const int grid = std::min(p.n_items, sms);
  kernel<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(tq, tk, tv, p);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "paged prefill launch");
  return B300ATTN_OK;
}

// FP8 prefill (d = 128, dense): q8 [B*N, Hq, 128] and k8 [B*N, Hkv, 128]
// e4m3 seen as [rows, heads, d] with one 128-byte box per row; v8t
// [B*Hkv, 128, Np] with boxes of 128 keys x all of d.
int launch_prefill_fp8(const void* q8, const void* k8, const void* v8t, int Np,
                       const PrefillParams& p, cudaStream_t stream) {
  using C = PrefillCfg<128, true>;
  CUtensorMap tq, tk, tv;
  int rc;
  if ((rc = make_map_3d(&tq, q8, 128, p.Hq, p.total_rows, 128, 1, C::BM,
                        CU_TENSOR_MAP_SWIZZLE_128B, "q8", true)) != B300ATTN_OK)
    return rc;
  if ((rc = make_map_3d(&tk, k8, 128, p.Hkv, p.total_rows, 128, 1, C::BN,
                        CU_TENSOR_MAP_SWIZZLE_128B, "k8", true)) != B300ATTN_OK)
    return rc;
  if ((rc = make_map_3d(&tv, v8t, Np, 128, static_cast<uint64_t>(p.B) * p.Hkv, C::BN, 128, 1,
                        CU_TENSOR_MAP_SWIZZLE_128B, "v8t", true)) != B300ATTN_OK)
    return rc;
  auto kernel = prefill_kernel<128, false, true>;
  if ((rc = set_smem(kernel, C::SMEM_BYTES)) != B300ATTN_OK) return rc;
  int sms = 0;
  if ((rc = sm_count(&sms)) != B300ATTN_OK) return rc;
  const int grid = std::min(p.n_items, sms);
  kernel<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(tq, tk, tv, p);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "FP8 prefill launch");
  return B300ATTN_OK;
}

int fp8_padded_len(int N) { return (N + 15) / 16 * 16; }

template <int D, int GT>
int launch_decode(const void* k_cache, const void* v_cache, const DecodeParams& p,
                  cudaStream_t stream) {
  using L = DecSmem<D, GT>;
  CUtensorMap tk, tv;
  int rc;
  // dense [B, Lmax, Hkv, D] or paged [num_pages, page_size, Hkv, D]
  const uint64_t rows = p.block_table ? p.page_size : p.Lmax;
  const uint64_t outer = p.block_table ? p.num_pages : p.B;
  if ((rc = make_map_4d(&tk, k_cache, D, p.Hkv, rows, outer, D, 1, kDecSub, 1,
                        CU_TENSOR_MAP_SWIZZLE_NONE, "k_cache")) != B300ATTN_OK)
    return rc;
  if ((rc = make_map_4d(&tv, v_cache, D, p.Hkv, rows, outer, D, 1, kDecSub, 1,
                        CU_TENSOR_MAP_SWIZZLE_NONE, "v_cache")) != B300ATTN_OK)
    return rc;
  if ((rc = set_smem(decode_partial_kernel<D, GT>, L::BYTES)) != B300ATTN_OK) return rc;
  const dim3 grid(p.S, p.Hkv * (p.G / GT), p.B);
  decode_partial_kernel<D, GT><<<grid, kDecThreads, L::BYTES, stream>>>(tk, tv, p);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return B300ATTN_OK;
}

template <int D>
int launch_decode_gt(int GT, const void* kc, const void* vc, const DecodeParams& p,
                     cudaStream_t s) {
  switch (GT) {
    case 8: return launch_decode<D, 8>(kc, vc, p, s);
    case 4: return launch_decode<D, 4>(kc, vc, p, s);
    case 2: return launch_decode<D, 2>(kc, vc, p, s);
    default: return launch_decode<D, 1>(kc, vc, p, s);
  }
}

// Many partials: one thread-block cluster of C CTAs per row, C = ceil(S / 256)
// capped at 8 (a CTA merges at most 256 partials, 16 per warp of 16 warps).
// Few partials (S <= 64): one warp per row.  With `dependent` the launch is
// programmatic: it may start while the preceding decode grid still runs, and
// waits in the kernel for that grid's partials.
template <int D>
int launch_combine_t(const float* pm, const float* pl, const float* po, void* o, float* lse,
                     int rows, int S, int o_f32, bool dependent, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  int na = 0;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  if (dependent) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cudaError_t e;
  if (S <= 64) {
    cfg.gridDim = dim3(static_cast<unsigned>((rows + 3) / 4), 1, 1);
    cfg.blockDim = dim3(128, 1, 1);
    cfg.attrs = attr;
    cfg.numAttrs = na;
    e = cudaLaunchKernelEx(&cfg, lse_combine_rows_kernel<D>, pm, pl, po, o, lse, rows, S, o_f32);
  } else {
    const int C = std::min(kCombMaxCluster, std::max(1, (S + 255) / 256));
    if (static_cast<long long>(rows) * C > 0x7fffffffLL)
      return fail(B300ATTN_ERR_UNSUPPORTED, "too many rows for one combine launch");
    cfg.gridDim = dim3(static_cast<unsigned>(rows * C), 1, 1);
    cfg.blockDim = dim3(16 * 32, 1, 1);
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = C;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
    cfg.attrs = attr;
    cfg.numAttrs = na;
    e = cudaLaunchKernelEx(&cfg, lse_combine_kernel<D, 16>, pm, pl, po, o, lse, S, o_f32);
  }
  if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  return B300ATTN_OK;
}

int launch_combine(const float* pm, const float* pl, const float* po, void* o, float* lse,
                   int rows, int S, int d, int o_f32, cudaStream_t stream,
                   bool dependent = false) {
  return d == 128 ? launch_combine_t<128>(pm, pl, po, o, lse, rows, S, o_f32, dependent, stream)
                  : launch_combine_t<64>(pm, pl, po, o, lse, rows, S, o_f32, dependent, stream);
}

// Number of 64-partial segments of the decode's two-level merge (0: one level).
int combine_segments(int S) { return S > 64 ? (S + kCombSeg - 1) / kCombSeg : 0; }

// The decode's merge: with more than 64 partials per row, segments of 64 are
// merged first into the workspace's second-level arrays (many small CTAs, all
// resident at once), then the segment triples by one warp per row.  Both
// launches are programmatic (they overlap the end of the grid before them).
template <int D>
int launch_decode_combine_t(const DecodeParams& p, void* o, float* lse, int o_f32,
                            cudaStream_t stream) {
  const int rows = p.B * p.Hq;
  const int nseg = combine_segments(p.S);
  if (nseg == 0)
    return launch_combine_t<D>(p.part_m, p.part_l, p.part_o, o, lse, rows, p.S, o_f32, true,
                               stream);
  if (rows > 65535) return fail(B300ATTN_ERR_UNSUPPORTED, "B*Hq=%d rows > 65535", rows);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(nseg), static_cast<unsigned>(rows), 1);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, lse_combine_segments_kernel<D>, p.part_m,
                                           p.part_l, p.part_o, p.seg_m, p.seg_l, p.seg_o, p.S,
                                           nseg);
  if (e != cudaSuccess) return cuda_fail(e, "combine (segments) launch");
  return launch_combine_t<D>(p.seg_m, p.seg_l, p.seg_o, o, lse, rows, nseg, o_f32, true, stream);
}

int launch_decode_combine(const DecodeParams& p, int d, void* o, float* lse, int o_f32,
                          cudaStream_t stream) {
  return d == 128 ? launch_decode_combine_t<128>(p, o, lse, o_f32, stream)
                  : launch_decode_combine_t<64>(p, o, lse, o_f32, stream);
}

template <int D>
int launch_backward(const void* q, const void* k, const void* v, const BwdParams& p,
                    cudaStream_t stream) {
  using C = BwdCfg<D>;
  CUtensorMap tq, tk, tv, tdo;
  int rc;
  if ((rc = make_map_4d(&tq, q, D, p.Hq, p.N, p.B, 64, 1, 128, 1, CU_TENSOR_MAP_SWIZZLE_128B,
                        "q")) != B300ATTN_OK)
    return rc;
  if ((rc = make_map_4d(&tk, k, D, p.Hkv, p.N, p.B, 64, 1, 128, 1, CU_TENSOR_MAP_SWIZZLE_128B,
                        "k")) != B300ATTN_OK)
    return rc;
  if ((rc = make_map_4d(&tv, v, D, p.Hkv, p.N, p.B, 64, 1, 128, 1, CU_TENSOR_MAP_SWIZZLE_128B,
                        "v")) != B300ATTN_OK)
    return rc;
  if ((rc = make_map_4d(&tdo, p.dO, D, p.Hq, p.N, p.B, 64, 1, 128, 1,
                        CU_TENSOR_MAP_SWIZZLE_128B, "dO")) != B300ATTN_OK)
    return rc;
  if ((rc = set_smem(bwd_dkdv_kernel<D>, DkdvSmem<D>::BYTES)) != B300ATTN_OK) return rc;
  if ((rc = set_smem(bwd_dq_kernel<D>, DqSmem<D>::BYTES)) != B300ATTN_OK) return rc;
  const long long rows = static_cast<long long>(p.B) * p.N * p.Hq;
  {
    constexpr long long per = bwd_preprocess_rows_per_cta<D>();
    bwd_preprocess_kernel<D><<<static_cast<unsigned>((rows + per - 1) / per), 256, 0, stream>>>(p);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "backward preprocess launch");
  const long long ntile = (p.N + 127) / 128;
  bwd_dkdv_kernel<D><<<static_cast<unsigned>(static_cast<long long>(p.B) * p.Hkv * ntile),
                       C::THREADS, DkdvSmem<D>::BYTES, stream>>>(tq, tk, tv, tdo, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "backward dK/dV launch");
  bwd_dq_kernel<D><<<static_cast<unsigned>(static_cast<long long>(p.B) * p.Hq * ntile),
                     C::THREADS, DqSmem<D>::BYTES, stream>>>(tq, tk, tv, tdo, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "backward dQ launch");
  return B300ATTN_OK;
}

int check_common(int d, int o_dtype) {
  if (d != 64 && d != 128)
    return fail(B300ATTN_ERR_UNSUPPORTED, "head dimension d=%d is not supported (64 or 128)", d);
  if (o_dtype != B300ATTN_BF16 && o_dtype != B300ATTN_F32)
    return fail(B300ATTN_ERR_INVALID, "o_dtype=%d must be 0 (bf16) or 1 (f32)", o_dtype);
  return B300ATTN_OK;
}

// Validates the decode arguments shared by attn_decode_partials and
// attn_decode_splitkv and fills `p`; returns B300ATTN_OK with p.B == 0 when
// there is nothing to compute.
int decode_setup(const void* q, const void* k_cache, const void* v_cache, const int* kv_len,
                 int B, int Hq, int Hkv, int max_kv_len, int d, float scale, int num_splits,
                 void* workspace, size_t workspace_bytes, DecodeParams& p, int& GT) {
  p.B = 0;
  if (B < 0 || Hq < 0 || Hkv < 0 || d < 0 || max_kv_len < 0)
    return fail(B300ATTN_ERR_INVALID, "negative size");
  if (B == 0 || Hq == 0) return B300ATTN_OK;
  if (Hkv == 0 || Hq % Hkv != 0)
    return fail(B300ATTN_ERR_INVALID, "Hq=%d must be a positive multiple of Hkv=%d", Hq, Hkv);
  int rc = check_common(d, B300ATTN_BF16);
  if (rc != B300ATTN_OK) return rc;
  if (max_kv_len < 1) return fail(B300ATTN_ERR_INVALID, "max_kv_len must be >= 1");
  if (num_splits < 1 || num_splits > 65535)
    return fail(B300ATTN_ERR_INVALID, "num_splits=%d must be in [1, 65535]", num_splits);
  if (B > 65535) return fail(B300ATTN_ERR_UNSUPPORTED, "B=%d > 65535", B);
  if (!q || !k_cache || !v_cache || !kv_len)
    return fail(B300ATTN_ERR_INVALID, "NULL tensor pointer");
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(B300ATTN_ERR_INVALID, "tensor pointers must be 16-byte aligned");
  if (!std::isfinite(scale) || scale < 0.f)
    return fail(B300ATTN_ERR_INVALID, "scale must be finite and >= 0");
  const size_t need = attn_decode_workspace_size(B, Hq, num_splits, d);
  if (!workspace || workspace_bytes < need)
    return fail(B300ATTN_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                workspace ? workspace_bytes : static_cast<size_t>(0));
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(B300ATTN_ERR_INVALID, "workspace must be 256-byte aligned");
  const int G = Hq / Hkv;
  GT = (G % 8 == 0) ? 8 : (G % 4 == 0) ? 4 : (G % 2 == 0) ? 2 : 1;
  if (static_cast<long long>(Hkv) * (G / GT) > 65535)
    return fail(B300ATTN_ERR_UNSUPPORTED, "too many heads for one launch");

  const size_t rows = static_cast<size_t>(B) * Hq * num_splits;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.kv_len = kv_len;
  char* ws = static_cast<char*>(workspace);
  p.part_m = reinterpret_cast<float*>(ws);
  p.part_l = reinterpret_cast<float*>(ws + align256(rows * 4));
  p.part_o = reinterpret_cast<float*>(ws + 2 * align256(rows * 4));
  // second-level triples of the two-level merge, after the partials
  const size_t srows = static_cast<size_t>(B) * Hq * combine_segments(num_splits);
  char* lvl2 = ws + 2 * align256(rows * 4) + align256(rows * d * 4);
  p.seg_m = reinterpret_cast<float*>(lvl2);
  p.seg_l = reinterpret_cast<float*>(lvl2 + align256(srows * 4));
  p.seg_o = reinterpret_cast<float*>(lvl2 + 2 * align256(srows * 4));
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Lmax = max_kv_len;
  p.chunk = attn_decode_chunk(max_kv_len, num_splits);
  p.S = num_splits;
  p.G = G;
  p.scale_log2 = scale * kLog2e;
  p.block_table = nullptr;
  p.page_size = 0;
  p.pages_per_seq = 0;
  p.num_pages = 0;
  return B300ATTN_OK;
}

int launch_partials(int d, int GT, const void* k_cache, const void* v_cache,
                    const DecodeParams& p, cudaStream_t stream) {
  return d == 128 ? launch_decode_gt<128>(GT, k_cache, v_cache, p, stream)
                  : launch_decode_gt<64>(GT, k_cache, v_cache, p, stream);
}
// ---------------------------------------------------------------------------
// Built-in scratch for attn_decode_splitkv_noalloc.  The split partials of
// that entry point live in this file-scope device array instead of a
// caller-supplied workspace.  Every device that loads this library holds the
// array for the life of the process.  Calls share it, so calls that overlap on
// the GPU race.  Nothing in it has to start at zero: the partial kernel writes
// every (m, l, o) triple, including the empty ones, before the combine reads
// it.
// ---------------------------------------------------------------------------
constexpr size_t kNoAllocScratchBytes = size_t(40) << 20;  // 40 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device.  In host code
// the array's name only stands in for the symbol, so the address is looked up
// with cudaGetSymbolAddress, once per device, on the first call made with that
// device current, and cached.
int noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices)
    return fail(B300ATTN_ERR_UNSUPPORTED, "device ordinal %d is out of range", dev);
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(g_noalloc_scratch)");
    if (!ptr) return fail(B300ATTN_ERR_CUDA, "cudaGetSymbolAddress returned NULL");
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return B300ATTN_OK;
}

// Self-test of the failure path: one thread waits on an mbarrier that nothing
// ever arrives on, with no copy or MMA in flight, so the bounded wait must run
// out after `limit_ns` and record its bit; the CTA then returns normally.
__device__ unsigned int g_selftest_status;
constexpr unsigned kStatusSelftest = 1u;

__global__ void __launch_bounds__(32) selftest_wait_kernel(unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, &g_selftest_status, kStatusSelftest, limit_ns);
}

}  // namespace

extern "C" {

int attn_version(void) { return 100; }

const char* attn_last_error(void) { return g_last_error.c_str(); }

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
             int Hkv, int N, int d, int causal, int window, float scale, cudaStream_t stream,
             int o_dtype) {
  if (B < 0 || Hq < 0 || Hkv < 0 || N < 0 || d < 0)
    return fail(B300ATTN_ERR_INVALID, "negative size (B=%d Hq=%d Hkv=%d N=%d d=%d)", B, Hq, Hkv,
                N, d);
  if (B == 0 || N == 0 || Hq == 0) return B300ATTN_OK;
  if (Hkv == 0 || Hq % Hkv != 0)
    return fail(B300ATTN_ERR_INVALID, "Hq=%d must be a positive multiple of Hkv=%d", Hq, Hkv);
  int rc = check_common(d, o_dtype);
  if (rc != B300ATTN_OK) return rc;
  if (!q || !k || !v || !o || !lse) return fail(B300ATTN_ERR_INVALID, "NULL tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return fail(B300ATTN_ERR_INVALID, "tensor pointers must be 16-byte aligned");
  if (causal != 0 && causal != 1) return fail(B300ATTN_ERR_INVALID, "causal must be 0 or 1");
  if (!std::isfinite(scale) || scale < 0.f)
    return fail(B300ATTN_ERR_INVALID, "scale must be finite and >= 0 (got %g)",
                static_cast<double>(scale));
  if (static_cast<long long>(B) * N > 0x7fffffffLL)
    return fail(B300ATTN_ERR_UNSUPPORTED, "B*N=%lld rows exceed 2^31-1",
                static_cast<long long>(B) * N);
  PrefillParams p{};
  p.o = o;
  p.lse = lse;
  p.cu_seqlens = nullptr;
  p.num_seqs = B;
  p.total_rows = B * N;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = N;
  p.causal = causal;
  p.window = window < 0 ? -1 : window;
  p.o_f32 = o_dtype == B300ATTN_F32;
  p.nqb = (N + 255) / 256;
  // a zero scale is kept strictly positive so that masked (-inf) scores stay -inf
  p.scale_log2 = std::fmax(scale * kLog2e, 1e-30f);
  const long long items = static_cast<long long>(p.nqb) * Hq * B;
  if (items > 0x7fffffffLL) return fail(B300ATTN_ERR_UNSUPPORTED, "too many query blocks");
  p.n_items = static_cast<int>(items);
  const long long q_tiles = static_cast<long long>(B) * Hq * ((N + 127) / 128);
  if (d == 64 && !causal && p.window >= 0 && p.window <= kBandMaxWindow &&
      q_tiles <= 0x7fffffffLL)
    return launch_prefill_band(q, k, v, p, stream);
  return d == 128 ? launch_prefill<128>(q, k, v, p, p.n_items, stream)
                  : launch_prefill<64>(q, k, v, p, p.n_items, stream);
}

int attn_fwd_paged(const void* q, const void* k_pages, const void* v_pages,
                   const int* block_table, void* o, float* lse, int B, int Hq, int Hkv, int N,
                   int d, int page_size, int num_pages, int pages_per_seq, int causal,
                   int window, float scale, cudaStream_t stream, int o_dtype) {
  if (B < 0 || Hq < 0 || Hkv < 0 || N < 0 || d < 0 || page_size < 0 || num_pages < 0 ||
      pages_per_seq < 0)
    return fail(B300ATTN_ERR_INVALID, "negative size");
  if (B == 0 || N == 0 || Hq == 0) return B300ATTN_OK;
  if (Hkv == 0 || Hq % Hkv != 0)
    return fail(B300ATTN_ERR_INVALID, "Hq=%d must be a positive multiple of Hkv=%d", Hq, Hkv);
  int rc = check_common(d, o_dtype);
  if (rc != B300ATTN_OK) return rc;
  if (page_size < 64 || page_size % 64 != 0)
    return fail(B300ATTN_ERR_UNSUPPORTED, "page_size=%d must be a positive multiple of 64",
                page_size);
  if (num_pages < 1 || pages_per_seq < 1)
    return fail(B300ATTN_ERR_INVALID, "num_pages and pages_per_seq must be >= 1");
  if (static_cast<long long>(pages_per_seq) * page_size < N)
    return fail(B300ATTN_ERR_INVALID, "pages_per_seq * page_size = %lld < N = %d",
                static_cast<long long>(pages_per_seq) * page_size, N);
  if (!q || !k_pages || !v_pages || !block_table || !o || !lse)
    return fail(B300ATTN_ERR_INVALID, "NULL tensor pointer");
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(o) ||
      !aligned16(lse))
    return fail(B300ATTN_ERR_INVALID, "tensor pointers must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(block_table) & 3u) != 0)
    return fail(B300ATTN_ERR_INVALID, "block_table must be 4-byte aligned");
  if (causal != 0 && causal != 1) return fail(B300ATTN_ERR_INVALID, "causal must be 0 or 1");
  if (!std::isfinite(scale) || scale < 0.f)
    return fail(B300ATTN_ERR_INVALID, "scale must be finite and >= 0 (got %g)",
                static_cast<double>(scale));
  if (static_cast<long long>(B) * N > 0x7fffffffLL)
    return fail(B300ATTN_ERR_UNSUPPORTED, "B*N=%lld rows exceed 2^31-1",
                static_cast<long long>(B) * N);
  PrefillParams p{};
  p.o = o;
  p.lse = lse;
  p.cu_seqlens = nullptr;
  p.num_seqs = B;
  p.total_rows = B * N;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = N;
  p.causal = causal;
  p.window = window < 0 ? -1 : window;
  p.o_f32 = o_dtype == B300ATTN_F32;
  p.nqb = (N + 255) / 256;
  p.scale_log2 = std::fmax(scale * kLog2e, 1e-30f);
  p.block_table = block_table;
  p.page_size = page_size;
  p.pages_per_seq = pages_per_seq;
  p.num_pages = num_pages;
  const long long items = static_cast<long long>(p.nqb) * Hq * B;
  if (items > 0x7fffffffLL) return fail(B300ATTN_ERR_UNSUPPORTED, "too many query blocks");
  p.n_items = static_cast<int>(items);
  return d == 128 ? launch_prefill_paged<128>(q, k_pages, v_pages, p, stream)
                  : launch_prefill_paged<64>(q, k_pages, v_pages, p, stream);
}

int attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                    const int* cu_seqlens, int num_seqs, int total_rows, int max_seqlen, int Hq,
                    int Hkv, int d, int causal, int window, float scale, cudaStream_t stream,
                    int o_dtype) {
  if (num_seqs < 0 || total_rows < 0 || max_seqlen < 0 || Hq < 0 || Hkv < 0 || d < 0)
    return fail(B300ATTN_ERR_INVALID, "negative size");
  if (num_seqs == 0 || total_rows == 0 || max_seqlen == 0 || Hq == 0) return B300ATTN_OK;
  if (num_seqs > kMaxVarlenSeqs)
    return fail(B300ATTN_ERR_UNSUPPORTED, "num_seqs=%d exceeds %d sequences per launch", num_seqs,
                kMaxVarlenSeqs);
  if (Hkv == 0 || Hq % Hkv != 0)
    return fail(B300ATTN_ERR_INVALID, "Hq=%d must be a positive multiple of Hkv=%d", Hq, Hkv);
  int rc = check_common(d, o_dtype);
  if (rc != B300ATTN_OK) return rc;
  if (!q || !k || !v || !o || !lse || !cu_seqlens)
    return fail(B300ATTN_ERR_INVALID, "NULL tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return fail(B300ATTN_ERR_INVALID, "tensor pointers must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) != 0)
    return fail(B300ATTN_ERR_INVALID, "cu_seqlens must be 4-byte aligned");
  if (causal != 0 && causal != 1) return fail(B300ATTN_ERR_INVALID, "causal must be 0 or 1");
  if (!std::isfinite(scale) || scale < 0.f)
    return fail(B300ATTN_ERR_INVALID, "scale must be finite and >= 0 (got %g)",
                static_cast<double>(scale));
  PrefillParams p{};
  p.o = o;
  p.lse = lse;
  p.cu_seqlens = cu_seqlens;
  p.num_seqs = num_seqs;
  p.total_rows = total_rows;
  p.B = 0;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = 0;
  p.causal = causal;
  p.window = window < 0 ? -1 : window;
  p.o_f32 = o_dtype == B300ATTN_F32;
  p.nqb = 0;
  p.n_items = 0;  // counted on the device from cu_seqlens
  p.scale_log2 = std::fmax(scale * kLog2e, 1e-30f);
  const long long bound =
      static_cast<long long>(num_seqs) * ((std::min(max_seqlen, total_rows) + 255) / 256) * Hq;
  if (bound > 0x7fffffffLL) return fail(B300ATTN_ERR_UNSUPPORTED, "too many query blocks");
  return d == 128 ? launch_prefill<128>(q, k, v, p, bound, stream)
                  : launch_prefill<64>(q, k, v, p, bound, stream);
}

size_t attn_fp8_workspace_size(int B, int Hkv, int N) {
  if (B <= 0 || Hkv <= 0 || N <= 0) return 256;
  return align256(static_cast<size_t>(B) * Hkv * ((N + 127) / 128) * sizeof(float));
}

int attn_fp8_padded_len(int N) { return N <= 0 ? 0 : fp8_padded_len(N); }

int attn_fp8_quantize(const void* q, const void* k, const void* v, void* q8, void* k8, void* v8t,
                      int* q_exp, int* k_exp, int* v_exp, int B, int Hq, int Hkv, int N, int d,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (B < 0 || Hq < 0 || Hkv < 0 || N < 0 || d < 0)
    return fail(B300ATTN_ERR_INVALID, "negative size (B=%d Hq=%d Hkv=%d N=%d d=%d)", B, Hq, Hkv,
                N, d);
  if (B == 0 || N == 0 || Hq == 0) return B300ATTN_OK;
  if (Hkv == 0 || Hq % Hkv != 0)
    return fail(B300ATTN_ERR_INVALID, "Hq=%d must be a positive multiple of Hkv=%d", Hq, Hkv);
  if (d != 128)
    return fail(B300ATTN_ERR_UNSUPPORTED, "FP8 path: head dimension d=%d is not supported (128)",
                d);
  if (!q || !k || !v || !q8 || !k8 || !v8t || !q_exp || !k_exp || !v_exp)
    return fail(B300ATTN_ERR_INVALID, "NULL tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(q8) || !aligned16(k8) ||
      !aligned16(v8t))
    return fail(B300ATTN_ERR_INVALID, "tensor pointers must be 16-byte aligned");
  if (static_cast<long long>(B) * N > 0x7fffffffLL)
    return fail(B300ATTN_ERR_UNSUPPORTED, "B*N=%lld rows exceed 2^31-1",
                static_cast<long long>(B) * N);
  const size_t need = attn_fp8_workspace_size(B, Hkv, N);
  if (!workspace || workspace_bytes < need)
    return fail(B300ATTN_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                workspace ? workspace_bytes : static_cast<size_t>(0));
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(B300ATTN_ERR_INVALID, "workspace must be 256-byte aligned");
  Fp8QuantParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.v = static_cast<const __nv_bfloat16*>(v);
  p.q8 = static_cast<uint8_t*>(q8);
  p.k8 = static_cast<uint8_t*>(k8);
  p.v8t = static_cast<uint8_t*>(v8t);
  p.q_exp = q_exp;
  p.k_exp = k_exp;
  p.v_exp = v_exp;
  p.v_tile_amax = static_cast<float*>(workspace);
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = N;
  p.Np = fp8_padded_len(N);
  p.nt = (N + 127) / 128;
  if (p.nt > 65535 || Hkv > 65535 || B > 65535)
    return fail(B300ATTN_ERR_UNSUPPORTED, "grid too large");
  fp8_vamax_kernel<128><<<dim3(p.nt, Hkv, B), kFp8QuantThreads, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "FP8 V maximum launch");
  const long long jobs = static_cast<long long>(B) * p.nt * (Hq + 2LL * Hkv);
  if (jobs > 0x7fffffffLL) return fail(B300ATTN_ERR_UNSUPPORTED, "too many tiles");
  fp8_quantize_kernel<128><<<static_cast<unsigned>(jobs), kFp8QuantThreads, 0, stream>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "FP8 quantize launch");
  return B300ATTN_OK;
}

int attn_fwd_fp8(const void* q8, const void* k8, const void* v8t, const int* q_exp,
                 const int* k_exp, const int* v_exp, void* o, float* lse, int B, int Hq, int Hkv,
                 int N, int d, int causal, int window, float scale, cudaStream_t stream,
                 int o_dtype) {
  if (B < 0 || Hq < 0 || Hkv < 0 || N < 0 || d < 0)
    return fail(B300ATTN_ERR_INVALID, "negative size (B=%d Hq=%d Hkv=%d N=%d d=%d)", B, Hq, Hkv,
                N, d);
  if (B == 0 || N == 0 || Hq == 0) return B300ATTN_OK;
  if (Hkv == 0 || Hq % Hkv != 0)
    return fail(B300ATTN_ERR_INVALID, "Hq=%d must be a positive multiple of Hkv=%d", Hq, Hkv);
  if (d != 128)
    return fail(B300ATTN_ERR_UNSUPPORTED, "FP8 path: head dimension d=%d is not supported (128)",
                d);
  int rc = check_common(d, o_dtype);
  if (rc != B300ATTN_OK) return rc;
  if (!q8 || !k8 || !v8t || !q_exp || !k_exp || !v_exp || !o || !lse)
    return fail(B300ATTN_ERR_INVALID, "NULL tensor pointer");
  if (!aligned16(q8) || !aligned16(k8) || !aligned16(v8t) || !aligned16(o) || !aligned16(lse))
    return fail(B300ATTN_ERR_INVALID, "tensor pointers must be 16-byte aligned");
  if (causal != 0 && causal != 1) return fail(B300ATTN_ERR_INVALID, "causal must be 0 or 1");
  if (!std::isfinite(scale) || scale < 0.f)
    return fail(B300ATTN_ERR_INVALID, "scale must be finite and >= 0 (got %g)",
                static_cast<double>(scale));
  if (static_cast<long long>(B) * N > 0x7fffffffLL)
    return fail(B300ATTN_ERR_UNSUPPORTED, "B*N=%lld rows exceed 2^31-1",
                static_cast<long long>(B) * N);
  PrefillParams p{};
  p.o = o;
  p.lse = lse;
  p.cu_seqlens = nullptr;
  p.num_seqs = B;
  p.total_rows = B * N;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = N;
  p.causal = causal;
  p.window = window < 0 ? -1 : window;
  p.o_f32 = o_dtype == B300ATTN_F32;
  p.nqb = (N + 255) / 256;
  p.scale_log2 = std::fmax(scale * kLog2e, 1e-30f);
  p.q_exp = q_exp;
  p.k_exp = k_exp;
  p.v_exp = v_exp;
  p.nt = (N + 127) / 128;
  const long long items = static_cast<long long>(p.nqb) * Hq * B;
  if (items > 0x7fffffffLL) return fail(B300ATTN_ERR_UNSUPPORTED, "too many query blocks");
  p.n_items = static_cast<int>(items);
  return launch_prefill_fp8(q8, k8, v8t, fp8_padded_len(N), p, stream);
}

size_t attn_bwd_workspace_size(int B, int Hq, int N) {
  if (B < 0 || Hq < 0 || N < 0) return 0;
  return align256(static_cast<size_t>(B) * Hq * N * sizeof(float));
}

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* dO, void* dq, void* dk, void* dv, void* workspace,
             size_t workspace_bytes, int B, int Hq, int Hkv, int N, int d, int causal, int window,
             float scale, cudaStream_t stream, int o_dtype) {
  if (B < 0 || Hq < 0 || Hkv < 0 || N < 0 || d < 0)
    return fail(B300ATTN_ERR_INVALID, "negative size (B=%d Hq=%d Hkv=%d N=%d d=%d)", B, Hq, Hkv,
                N, d);
  if (B == 0 || N == 0 || Hq == 0) return B300ATTN_OK;
  if (Hkv == 0 || Hq % Hkv != 0)
    return fail(B300ATTN_ERR_INVALID, "Hq=%d must be a positive multiple of Hkv=%d", Hq, Hkv);
  int rc = check_common(d, o_dtype);
  if (rc != B300ATTN_OK) return rc;
  if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv)
    return fail(B300ATTN_ERR_INVALID, "NULL tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(dO) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return fail(B300ATTN_ERR_INVALID, "tensor pointers must be 16-byte aligned");
  if (causal != 0 && causal != 1) return fail(B300ATTN_ERR_INVALID, "causal must be 0 or 1");
  if (!std::isfinite(scale) || scale < 0.f)
    return fail(B300ATTN_ERR_INVALID, "scale must be finite and >= 0 (got %g)",
                static_cast<double>(scale));
  const size_t need = attn_bwd_workspace_size(B, Hq, N);
  if (!workspace || workspace_bytes < need)
    return fail(B300ATTN_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                workspace ? workspace_bytes : static_cast<size_t>(0));
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(B300ATTN_ERR_INVALID, "workspace must be 256-byte aligned");
  const long long ntile = (static_cast<long long>(N) + 127) / 128;
  if (static_cast<long long>(B) * Hq * ntile > 0x7fffffffLL ||
      static_cast<long long>(B) * N * Hq / 8 + 1 > 0x7fffffffLL)
    return fail(B300ATTN_ERR_UNSUPPORTED, "problem too large for one launch");
  BwdParams p;
  p.o = o;
  p.dO = static_cast<const __nv_bfloat16*>(dO);
  p.lse = lse;
  p.dvec = static_cast<float*>(workspace);
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.N = N;
  p.causal = causal;
  p.window = window < 0 ? -1 : window;
  p.o_f32 = o_dtype == B300ATTN_F32;
  p.scale = scale;
  p.scale_log2 = std::fmax(scale * kLog2e, 1e-30f);
  return d == 128 ? launch_backward<128>(q, k, v, p, stream)
                  : launch_backward<64>(q, k, v, p, stream);
}

int attn_decode_chunk(int max_kv_len, int num_splits) {
  if (max_kv_len < 1 || num_splits < 1)
    return fail(B300ATTN_ERR_INVALID, "max_kv_len=%d and num_splits=%d must be >= 1", max_kv_len,
                num_splits);
  const long long c = (static_cast<long long>(max_kv_len) + num_splits - 1) / num_splits;
  return static_cast<int>((c + kDecSub - 1) / kDecSub * kDecSub);
}

size_t attn_decode_workspace_size(int B, int Hq, int num_splits, int d) {
  if (B < 0 || Hq < 0 || num_splits < 1 || d < 1) return 0;
  const size_t rows = static_cast<size_t>(B) * Hq * num_splits;
  const size_t srows = static_cast<size_t>(B) * Hq * combine_segments(num_splits);
  return 2 * align256(rows * sizeof(float)) + align256(rows * d * sizeof(float)) +
         (srows ? 2 * align256(srows * sizeof(float)) + align256(srows * d * sizeof(float)) : 0);
}


int attn_decode_partials(const void* q, const void* k_cache, const void* v_cache,
                         const int* kv_len, int B, int Hq, int Hkv, int max_kv_len, int d,
                         float scale, int num_splits, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream) {
  DecodeParams p;
  int GT = 1;
  int rc = decode_setup(q, k_cache, v_cache, kv_len, B, Hq, Hkv, max_kv_len, d, scale,
                        num_splits, workspace, workspace_bytes, p, GT);
  if (rc != B300ATTN_OK || p.B == 0) return rc;
  return launch_partials(d, GT, k_cache, v_cache, p, stream);
}

int attn_decode_splitkv(const void* q, const void* k_cache, const void* v_cache,
                        const int* kv_len, void* o, float* lse, int B, int Hq, int Hkv,
                        int max_kv_len, int d, float scale, int num_splits, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream, int o_dtype) {
  DecodeParams p;
  int GT = 1;
  int rc = decode_setup(q, k_cache, v_cache, kv_len, B, Hq, Hkv, max_kv_len, d, scale,
                        num_splits, workspace, workspace_bytes, p, GT);
  if (rc != B300ATTN_OK || p.B == 0) return rc;
  if ((rc = check_common(d, o_dtype)) != B300ATTN_OK) return rc;
  if (!o || !lse) return fail(B300ATTN_ERR_INVALID, "NULL tensor pointer");
  if (!aligned16(o) || !aligned16(lse))
    return fail(B300ATTN_ERR_INVALID, "tensor pointers must be 16-byte aligned");
  if ((rc = launch_partials(d, GT, k_cache, v_cache, p, stream)) != B300ATTN_OK) return rc;
  return launch_decode_combine(p, d, o, lse, o_dtype == B300ATTN_F32, stream);
}

int attn_decode_splitkv_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                const int* kv_len, void* o, float* lse, int B, int Hq, int Hkv,
                                int max_kv_len, int d, float scale, int num_splits,
                                cudaStream_t stream, int o_dtype) {
  if (B < 0 || Hq < 0 || num_splits < 0 || d < 0)
    return fail(B300ATTN_ERR_INVALID, "negative size");
  if (B == 0 || Hq == 0) return B300ATTN_OK;
  const size_t need = attn_decode_workspace_size(B, Hq, num_splits, d);
  if (need > kNoAllocScratchBytes)
    return fail(B300ATTN_ERR_WORKSPACE,
                "attn_decode_splitkv_noalloc: B=%d Hq=%d num_splits=%d d=%d needs %zu bytes of "
                "split partials, more than the built-in scratch of %zu bytes; use "
                "attn_decode_splitkv with a workspace of your own",
                B, Hq, num_splits, d, need, kNoAllocScratchBytes);
  void* scratch = nullptr;
  int rc = noalloc_scratch(&scratch);
  if (rc != B300ATTN_OK) return rc;
  return attn_decode_splitkv(q, k_cache, v_cache, kv_len, o, lse, B, Hq, Hkv, max_kv_len, d,
                             scale, num_splits, scratch, kNoAllocScratchBytes, stream, o_dtype);
}

int attn_decode_splitkv_paged(const void* q, const void* k_pages, const void* v_pages,
                              const int* block_table, const int* kv_len, void* o, float* lse,
                              int B, int Hq, int Hkv, int page_size, int num_pages,
                              int pages_per_seq, int d, float scale, int num_splits,
                              void* workspace, size_t workspace_bytes, cudaStream_t stream,
                              int o_dtype) {
  if (page_size < 0 || num_pages < 0 || pages_per_seq < 0)
    return fail(B300ATTN_ERR_INVALID, "negative page geometry");
  if (B > 0 && Hq > 0) {
    if (page_size < kDecSub || page_size % kDecSub != 0)
      return fail(B300ATTN_ERR_UNSUPPORTED, "page_size=%d must be a positive multiple of %d",
                  page_size, kDecSub);
    if (num_pages < 1 || pages_per_seq < 1)
      return fail(B300ATTN_ERR_INVALID, "num_pages and pages_per_seq must be >= 1");
    if (!block_table) return fail(B300ATTN_ERR_INVALID, "NULL block_table");
    if ((reinterpret_cast<uintptr_t>(block_table) & 3u) != 0)
      return fail(B300ATTN_ERR_INVALID, "block_table must be 4-byte aligned");
  }
  const long long lmax = static_cast<long long>(pages_per_seq) * page_size;
  if (lmax > 0x7fffffffLL) return fail(B300ATTN_ERR_UNSUPPORTED, "sequence capacity too large");
  DecodeParams p;
  int GT = 1;
  int rc = decode_setup(q, k_pages, v_pages, kv_len, B, Hq, Hkv, static_cast<int>(lmax), d,
                        scale, num_splits, workspace, workspace_bytes, p, GT);
  if (rc != B300ATTN_OK || p.B == 0) return rc;
  if ((rc = check_common(d, o_dtype)) != B300ATTN_OK) return rc;
  if (!o || !lse) return fail(B300ATTN_ERR_INVALID, "NULL tensor pointer");
  if (!aligned16(o) || !aligned16(lse))
    return fail(B300ATTN_ERR_INVALID, "tensor pointers must be 16-byte aligned");
  // the chunk is a multiple of the 64-key stage, and so is page_size: no
  // stage straddles two pages
  p.block_table = block_table;
  p.page_size = page_size;
  p.pages_per_seq = pages_per_seq;
  p.num_pages = num_pages;
  if ((rc = launch_partials(d, GT, k_pages, v_pages, p, stream)) != B300ATTN_OK) return rc;
  return launch_decode_combine(p, d, o, lse, o_dtype == B300ATTN_F32, stream);
}

int lse_tree_combine(const float* part_m, const float* part_l, const float* part_o, void* o,
                     float* lse, int rows, int num_splits, int d, cudaStream_t stream,
                     int o_dtype) {
  if (rows < 0 || d < 0) return fail(B300ATTN_ERR_INVALID, "negative size");
  if (rows == 0) return B300ATTN_OK;
  int rc = check_common(d, o_dtype);
  if (rc != B300ATTN_OK) return rc;
  if (num_splits < 1) return fail(B300ATTN_ERR_INVALID, "num_splits must be >= 1");
  if (!part_m || !part_l || !part_o || !o || !lse)
    return fail(B300ATTN_ERR_INVALID, "NULL tensor pointer");
  if (!aligned16(part_o) || !aligned16(o))
    return fail(B300ATTN_ERR_INVALID, "part_o and o must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(part_m) & 3u) || (reinterpret_cast<uintptr_t>(part_l) & 3u) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return fail(B300ATTN_ERR_INVALID, "part_m, part_l and lse must be 4-byte aligned");
  return launch_combine(part_m, part_l, part_o, o, lse, rows, num_splits, d,
                        o_dtype == B300ATTN_F32, stream);
}

int attn_selftest_bounded_wait(unsigned long long limit_ns, cudaStream_t stream) {
  if (limit_ns < 1000ull || limit_ns > 100000000ull)
    return fail(B300ATTN_ERR_INVALID, "limit_ns=%llu must lie in [1e3, 1e8] (1 us .. 100 ms)",
                limit_ns);
  selftest_wait_kernel<<<1, 32, 0, stream>>>(limit_ns);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return B300ATTN_OK;
}

int attn_device_status(cudaStream_t stream) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned int a = 0, b = 0, c = 0, t = 0, dbg = 0;
  const unsigned int zero = 0;
  if ((e = cudaMemcpyFromSymbol(&a, g_prefill_status, sizeof(a))) != cudaSuccess ||
      (e = cudaMemcpyFromSymbol(&b, g_decode_status, sizeof(b))) != cudaSuccess ||
      (e = cudaMemcpyFromSymbol(&c, g_bwd_status, sizeof(c))) != cudaSuccess ||
      (e = cudaMemcpyFromSymbol(&t, g_selftest_status, sizeof(t))) != cudaSuccess ||
      (e = cudaMemcpyFromSymbol(&dbg, g_debug_status, sizeof(dbg))) != cudaSuccess)
    return cuda_fail(e, "reading the device status word");
  if (dbg) {  // debug build only: a device-side check failed
    cudaMemcpyToSymbol(g_debug_status, &zero, sizeof(zero));
    if ((a | b | c | t) == 0)
      return fail(B300ATTN_ERR_INVALID,
                  "debug build: a device-side check failed (bits 0x%x: 1 kv_len outside "
                  "[0, max_kv_len], 2 cu_seqlens not monotone or outside [0, total_rows], "
                  "4/8/16/32/64 a prefill item, band tile, decode split, backward tile or "
                  "FP8 tile outside the launch)",
                  dbg);
  }
  if (a | b | c | t) {
    cudaMemcpyToSymbol(g_prefill_status, &zero, sizeof(zero));
    cudaMemcpyToSymbol(g_decode_status, &zero, sizeof(zero));
    cudaMemcpyToSymbol(g_bwd_status, &zero, sizeof(zero));
    cudaMemcpyToSymbol(g_selftest_status, &zero, sizeof(zero));
    if ((a & ~kStatusPrefillBadPage) == 0 && (c | t) == 0 && (b & ~kStatusDecodeBadPage) == 0)
      return fail(B300ATTN_ERR_INVALID,
                  "a paged call met a block_table entry outside [0, num_pages) (prefill bits "
                  "0x%x, decode bits 0x%x); those keys were left out of the result",
                  a, b);
    return fail(B300ATTN_ERR_TIMEOUT,
                "a kernel gave up on a bounded wait (status bits prefill=0x%x decode=0x%x "
                "backward=0x%x self-test=0x%x)",
                a, b, c, t);
  }
  return B300ATTN_OK;
}

}  // extern "C"
