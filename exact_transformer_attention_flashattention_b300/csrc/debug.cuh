// Debug checks, compiled in only with -DB300ATTN_DEBUG (libb300attn_debug.so).
//
// The release build clamps caller data that could send a kernel out of range
// (kv_len to [0, max_kv_len], cu_seqlens into [0, total_rows]) and relies on
// internal index invariants.  The debug build also checks them on the device:
// a failed check ORs a bit into g_debug_status and the kernel carries on with
// the clamped values (no trap, no early exit, no wait), so a misuse is
// reported by attn_device_status instead of being absorbed silently.  In a
// release build B300_DCHECK compiles to nothing and the kernels are unchanged.
#pragma once

namespace b300 {

__device__ unsigned int g_debug_status;  // OR of kDbg* bits (debug build only)

constexpr unsigned kDbgKvLen = 1u;         // decode: kv_len[b] outside [0, max_kv_len]
constexpr unsigned kDbgCuSeqlens = 2u;     // varlen prefill: cu_seqlens not monotone or outside [0, total_rows]
constexpr unsigned kDbgPrefillItem = 4u;   // prefill: work item outside its sequence, head or key range
constexpr unsigned kDbgBandTile = 8u;      // band prefill: Q tile outside the launch
constexpr unsigned kDbgDecodeSplit = 16u;  // decode: split, head group or sequence outside the grid's shape
constexpr unsigned kDbgBwdTile = 32u;      // backward: tile or head outside the launch
constexpr unsigned kDbgFp8Job = 64u;       // FP8 quantisation: tile outside the launch

}  // namespace b300

#ifdef B300ATTN_DEBUG
#define B300_DCHECK(cond, bit)                                   \
  do {                                                           \
    if (!(cond)) atomicOr(&::b300::g_debug_status, (bit));       \
  } while (0)
#else
#define B300_DCHECK(cond, bit) \
  do {                         \
  } while (0)
#endif
