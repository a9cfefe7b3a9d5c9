// debug_checks.cuh -- device-side bounds checks of the debug build.
//
// Compiled with -DJVP_DEBUG_CHECKS (build.build(debug=True)), every
// hand-computed TMEM column range, shared-memory offset and global row or
// column index of the tensor-core kernels is checked before the access it
// guards.  A failed check skips that access (no trap) and sets bit 1 of the
// library's device status word plus bit (8 + site) naming the kind of index;
// jvp_attn_get_device_status() then reports JVP_ERR_BOUNDS.  In the ordinary
// build JVP_CHECK is the constant true and the checks compile away.
#pragma once

namespace jvp {

enum CheckSite : unsigned {
  kChkTmem = 0,       // TMEM column range of a tcgen05.ld / st / mma
  kChkSmem = 1,       // shared-memory offset of a staged row or received state
  kChkGlobalRow = 2,  // global row index (lse, mu, per-row scalars, workspace rows)
  kChkGlobalCol = 3,  // global column index of a stored row piece
};

#ifdef JVP_DEBUG_CHECKS
__device__ __forceinline__ bool debug_check(bool ok, unsigned int* status, unsigned site) {
  if (!ok) atomicOr(status, 2u | (1u << (8u + site)));
  return ok;
}
#define JVP_CHECK(cond, status, site) (::jvp::debug_check((cond), (status), (site)))
#else
#define JVP_CHECK(cond, status, site) (true)
#endif

}  // namespace jvp
