// Shared device helpers of libpkv: status word, bf16 bit handling, mbarrier,
// bulk-async and tensor (TMA) copies.  Inline PTX written from the PTX ISA
// description of each instruction; sm_100-family only.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pkv.h"

#define PKV_DEVINL __device__ __forceinline__

namespace pkv {

// Kernels receive the address of the library's device status word and record
// the first error they see there (0 = none); pkv_read_device_status reads it.
PKV_DEVINL void raise_status(int* status, int code) { atomicCAS(status, 0, code); }

// Wait budget of a pipeline wait before it gives up and raises PKV_ERR_TIMEOUT.
constexpr unsigned long long kWaitBudgetNs = 2000000000ull;  // 2 s

PKV_DEVINL unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

PKV_DEVINL uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ bf16 bits
PKV_DEVINL float bf16lo_to_f32(uint32_t w) { return __uint_as_float(w << 16); }
PKV_DEVINL float bf16hi_to_f32(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Round-to-nearest-even fp32 -> bf16 pair (lo in bits 0..15), via the hardware cvt.
PKV_DEVINL uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// ------------------------------------------------------------------ mbarrier
PKV_DEVINL void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

PKV_DEVINL void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

PKV_DEVINL void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

PKV_DEVINL void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Predicated forms for converged warps: every lane executes the instruction and only
// lanes with `on` perform it, so a single-lane action needs no branch (reconverging a
// diverged warp costs hundreds of cycles on a busy scheduler).
PKV_DEVINL void mbar_arrive_if(bool on, uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %1, 0;\n\t"
        "@q mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}" ::"r"(smem_u32(bar)),
        "r"(static_cast<uint32_t>(on))
        : "memory");
}

PKV_DEVINL void mbar_arrive_expect_tx_if(bool on, uint64_t* bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\t"
        "@q mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
        "r"(bytes), "r"(static_cast<uint32_t>(on))
        : "memory");
}

PKV_DEVINL bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for phase `parity` of `bar` to complete.  Returns false (and
// raises PKV_ERR_TIMEOUT) if it has not completed within kWaitBudgetNs.
PKV_DEVINL bool mbar_wait(uint64_t* bar, uint32_t parity, int* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > kWaitBudgetNs) {
            raise_status(status, PKV_ERR_TIMEOUT);
            return false;
        }
    }
}

// Bounded wait of a converged warp: every lane polls and a vote makes the outcome
// uniform (a completed phase stays completed), so the warp never diverges.
PKV_DEVINL bool mbar_wait_warp(uint64_t* bar, uint32_t parity, int* status) {
    if (__any_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (;;) {
        if (__any_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
        if (__any_sync(0xffffffffu, globaltimer_ns() - t0 > kWaitBudgetNs)) {
            if ((threadIdx.x & 31) == 0) raise_status(status, PKV_ERR_TIMEOUT);
            __syncwarp();
            return false;
        }
    }
}

// ------------------------------------------------------------------ async copies
// 1-D bulk copy global -> shared, completion counted on `bar` (bytes % 16 == 0,
// both addresses 16-byte aligned).
PKV_DEVINL void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// L2 eviction priority of a copy (createpolicy): lines fetched under an evict-first
// policy are the first ones L2 gives up.  The decode kernels stream every K/V byte
// exactly once, so they copy under it and leave L2 to what is re-read (query rows,
// block tables, partials, a shared prefix): on the Llama-3-8B-shaped decode batch this
// took the step from 90.5 to 86.4 us.
PKV_DEVINL uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// bulk_g2s under an L2 cache policy.
PKV_DEVINL void bulk_g2s_hint(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar,
                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// 2-D tiled tensor copy global -> shared through a tensor map (coordinates in
// elements, innermost first).
PKV_DEVINL void tma_load_3d(void* smem_dst, const void* tmap, int32_t x, int32_t y, int32_t z,
                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(smem_dst)),
        "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

PKV_DEVINL void tma_load_2d_if(bool on, void* smem_dst, const void* tmap, int32_t x, int32_t y,
                               uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %5, 0;\n\t"
        "@q cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];\n\t}" ::"r"(smem_u32(smem_dst)),
        "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar)), "r"(static_cast<uint32_t>(on))
        : "memory");
}

PKV_DEVINL void tma_load_4d_if(bool on, void* smem_dst, const void* tmap, int32_t x, int32_t y,
                               int32_t z, int32_t w, uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %7, 0;\n\t"
        "@q cp.async.bulk.tensor.4d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];\n\t}" ::"r"(smem_u32(smem_dst)),
        "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar)),
        "r"(static_cast<uint32_t>(on))
        : "memory");
}

// tma_load_2d_if / tma_load_4d_if under an L2 cache policy.
PKV_DEVINL void tma_load_2d_hint_if(bool on, void* smem_dst, const void* tmap, int32_t x,
                                    int32_t y, uint64_t* bar, uint64_t policy) {
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %5, 0;\n\t"
        "@q cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %6;\n\t}" ::"r"(smem_u32(smem_dst)),
        "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar)), "r"(static_cast<uint32_t>(on)),
        "l"(policy)
        : "memory");
}

PKV_DEVINL void tma_load_4d_hint_if(bool on, void* smem_dst, const void* tmap, int32_t x,
                                    int32_t y, int32_t z, int32_t w, uint64_t* bar,
                                    uint64_t policy) {
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %7, 0;\n\t"
        "@q cp.async.bulk.tensor.4d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %8;\n\t}" ::"r"(smem_u32(smem_dst)),
        "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar)),
        "r"(static_cast<uint32_t>(on)), "l"(policy)
        : "memory");
}

PKV_DEVINL void prefetch_tmap(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// Generic-proxy shared-memory writes -> visible to the async proxy (tensor core).
PKV_DEVINL void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start before its predecessor on the stream finishes;
// griddep_wait() blocks until that predecessor has completed and its writes are
// visible (a no-op otherwise).  griddep_launch_dependents() lets the next such
// kernel be scheduled early.
PKV_DEVINL void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
PKV_DEVINL void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

PKV_DEVINL float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// max(a, b, c) in one instruction (sm_100+ three-input form).
PKV_DEVINL float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Packed pair arithmetic (sm_100+ f32x2): (d0, d1) = (a0 * b0 + c0, a1 * b1 + c1).
PKV_DEVINL void ffma2(float& d0, float& d1, float a0, float a1, float b0, float b1, float c0,
                      float c1) {
    asm("{\n\t.reg .b64 a, b, c, d;\n\t"
        "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %7};\n\t"
        "fma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
PKV_DEVINL void fadd2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 a, b, d;\n\t"
        "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "add.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// Upper 16 bits of a (low half of the result) and of b (high half): two fp32 values
// truncated to bf16 and packed, in one byte permute.
PKV_DEVINL uint32_t pack_bf16x2_trunc(float a, float b) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(r) : "r"(__float_as_uint(a)), "r"(__float_as_uint(b)));
    return r;
}

// One lane of the converged warp (the lowest active one) gets true.
PKV_DEVINL bool elect_one() {
    uint32_t p = 0;
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\tselp.u32 %0, 1, 0, e;\n\t}"
        : "=r"(p));
    return p != 0;
}

}  // namespace pkv
