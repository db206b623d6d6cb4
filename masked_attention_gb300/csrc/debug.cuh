// Device-side bounds checks of the debug build (compiled with -DMATTN_DEBUG
// into libmattn_debug.so; the release library compiles them away).
//
// Each index that a kernel computes for a global load or store outside the
// tensor-map copies (which the hardware clamps) goes through
// MATTN_IN_BOUNDS(site, index, bound). In the debug build an index outside
// [0, bound) is recorded in the translation unit's debug record (the first
// one: its site, index and bound; later ones only counted) and the access
// is skipped: a load reads 0, a store does not happen. Nothing traps, so the
// context stays usable and the host reads the record afterwards
// (attn_debug_record). In the release build the macro is the constant true.
#pragma once

#include <cstdint>

namespace mattn {

// Access sites; the host names them in attn_debug_site_name().
enum DebugSite : int {
  kSiteNone = 0,
  kSiteFwdList = 1,       // block-mask list entry (row order, counts, tile index)
  kSiteFwdPage = 2,       // page-table entry read by the forward
  kSiteFwdDoc = 3,        // document id read by the forward
  kSiteFwdO = 4,          // O row written by the forward
  kSiteFwdLse = 5,        // LSE written by the forward
  kSiteBwdList = 6,       // block-mask list entry read by the backward
  kSiteBwdRow = 7,        // row term (LSE, Delta) of the backward
  kSiteBwdDoc = 8,        // document id read by the backward
  kSiteBwdGrad = 9,       // dQ, dK or dV row written by the backward
  kSiteDecQ = 10,         // query row read by decode
  kSiteDecKV = 11,        // key/value row read by decode
  kSiteDecTable = 12,     // page-table entry read by decode
  kSiteDecSide = 13,      // document id or relative-bias entry read by decode
  kSiteDecOut = 14,       // O / LSE or a split's partial written by decode
  kSiteCombineIn = 15,    // part read by the merge
  kSiteCombineOut = 16,   // merged row written
  kSiteF32 = 17,          // any access of the fp32 forward
  kSiteMaskBuild = 18,    // block-mask list written by the builder
  kSiteSelfTest = 19,     // the planted index of attn_debug_selftest
  kSiteCount
};

struct DebugRecord {
  unsigned long long count;  // checks that failed
  int site;                  // DebugSite of the first failure
  int pad;
  long long index;           // its index
  long long bound;           // and the bound it broke
};

#ifdef MATTN_DEBUG

namespace {
// One record per translation unit (each unit is its own device module).
__device__ DebugRecord g_debug_record;
}  // namespace

__device__ __forceinline__ bool debug_in_bounds(int site, long long index, long long bound) {
  if (index >= 0 && index < bound) return true;
  if (atomicAdd(&g_debug_record.count, 1ull) == 0ull) {
    g_debug_record.site = site;
    g_debug_record.index = index;
    g_debug_record.bound = bound;
  }
  return false;
}

#define MATTN_IN_BOUNDS(site, index, bound) \
  (::mattn::debug_in_bounds((site), (long long)(index), (long long)(bound)))

// Host side of a translation unit's record: copy out and clear.
#define MATTN_DEBUG_RECORD_ACCESSORS(name)                                          \
  cudaError_t debug_fetch_##name(DebugRecord* out) {                                \
    return cudaMemcpyFromSymbol(out, g_debug_record, sizeof(DebugRecord));          \
  }                                                                                 \
  cudaError_t debug_clear_##name() {                                                \
    const DebugRecord zero{};                                                       \
    return cudaMemcpyToSymbol(g_debug_record, &zero, sizeof(DebugRecord));          \
  }

#else

#define MATTN_IN_BOUNDS(site, index, bound) true
#define MATTN_DEBUG_RECORD_ACCESSORS(name)

#endif

}  // namespace mattn
