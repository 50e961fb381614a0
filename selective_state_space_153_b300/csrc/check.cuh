// Checked build (-DSSM_CHECK): bounds checks on global and shared memory accesses and
// NaN-poisoned shared memory, in place of a memory checker. A failed check records
// SSM_ERR_CHECK in the device status word (read by ssm_stream_status) and the access is
// skipped (a load returns zero); nothing traps. In the normal build every check is the
// constant `true` and compiles away.
#pragma once
#include <stdint.h>

#include "ptx.cuh"

namespace ssm {

constexpr int kStatusCheck = 9;   // SSM_ERR_CHECK

#ifdef SSM_CHECK
// [p, p + n) inside [base, base + total): bytes
__device__ __forceinline__ bool chk_global(const void *base, uint64_t total, const void *p, uint64_t n) {
    const uint64_t b = reinterpret_cast<uint64_t>(base), a = reinterpret_cast<uint64_t>(p);
    const bool ok = base != nullptr && a >= b && a + n <= b + total;
    if (!ok) set_status(kStatusCheck);
    return ok;
}
__device__ __forceinline__ uint32_t dyn_smem_bytes() {
    uint32_t v;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(v));
    return v;
}
// [p, p + n) inside the CTA's dynamic shared memory starting at base
__device__ __forceinline__ bool chk_smem(const void *base, const void *p, uint64_t n) {
    const uint64_t b = reinterpret_cast<uint64_t>(base), a = reinterpret_cast<uint64_t>(p);
    const bool ok = a >= b && a + n <= b + dyn_smem_bytes();
    if (!ok) set_status(kStatusCheck);
    return ok;
}
// same for a 32-bit shared-space address (cp.async destinations)
__device__ __forceinline__ bool chk_smem_u32(uint32_t base, uint32_t addr, uint32_t n) {
    const bool ok = addr >= base && addr + n <= base + dyn_smem_bytes();
    if (!ok) set_status(kStatusCheck);
    return ok;
}
// every word of the dynamic shared memory set to a quiet NaN, so that a read of a word no
// thread wrote turns into NaN in the results
__device__ __forceinline__ void poison_smem(void *base) {
    uint32_t *w = reinterpret_cast<uint32_t *>(base);
    const uint32_t n = dyn_smem_bytes() / 4;
    for (uint32_t i = threadIdx.x; i < n; i += blockDim.x) w[i] = 0x7fc00000u;
    __syncthreads();
}
#define SSM_CHK_G(base, total, p, n) ::ssm::chk_global((base), (uint64_t)(total), (p), (uint64_t)(n))
#define SSM_CHK_S(base, p, n) ::ssm::chk_smem((base), (p), (uint64_t)(n))
#define SSM_CHK_SU(base, addr, n) ::ssm::chk_smem_u32((base), (addr), (n))
#define SSM_POISON_SMEM(base) ::ssm::poison_smem(base)
#else
#define SSM_CHK_G(base, total, p, n) true
#define SSM_CHK_S(base, p, n) true
#define SSM_CHK_SU(base, addr, n) true
#define SSM_POISON_SMEM(base) ((void)0)
#endif

}  // namespace ssm

namespace ssm {
// checked loads and stores: the access happens only when it passes the check (a failed load
// yields a zero value)
template <typename V>
__device__ __forceinline__ V ld_chk_s(const void *sbase, const V *p) {
    return SSM_CHK_S(sbase, p, sizeof(V)) ? *p : V{};
}
template <typename V>
__device__ __forceinline__ void st_chk_s(const void *sbase, V *p, const V &v) {
    if (SSM_CHK_S(sbase, p, sizeof(V))) *p = v;
}
template <typename V>
__device__ __forceinline__ V ld_chk_g(const void *gbase, uint64_t total, const V *p) {
    return SSM_CHK_G(gbase, total, p, sizeof(V)) ? *p : V{};
}
template <typename V>
__device__ __forceinline__ void st_chk_g(void *gbase, uint64_t total, V *p, const V &v) {
    if (SSM_CHK_G(gbase, total, p, sizeof(V))) *p = v;
}
}  // namespace ssm
