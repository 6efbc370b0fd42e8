// dv_common.cuh -- device helpers shared by the sm_103a kernels of libdv.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dv_internal.h"

namespace dv {

#define DV_DEV __device__ __forceinline__

constexpr int kWarp = 32;

// ---------------------------------------------------------------------------
// Global-memory access.
//
// Weights are read exactly once per call and never written: 16-byte vector
// loads through the non-coherent path, not allocated in L1, with a 256-byte
// L2 prefetch hint so DRAM sees whole bursts.
// The asm is volatile so a prefetch is issued where it is written (ahead of
// the arithmetic on the previous batch), not moved next to its first use.
DV_DEV uint4 ld_stream(const void *p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

// Data that a preceding kernel writes while this one may already be resident
// (programmatic dependent launch: the KV cache's appended slot): 16-byte loads
// at L2, never through the non-coherent read-only path, which is only valid
// for data that no grid writes during the reading kernel's lifetime.
DV_DEV uint4 ld_stream_coherent(const void *p)
{
    uint4 r;
    asm volatile("ld.global.cg.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// Values written by other CTAs of the same kernel: read at L2 (bypass L1).
DV_DEV float ld_cg(const float *p) { return __ldcg(p); }
DV_DEV int ld_cg(const int *p) { return __ldcg(p); }

// Record the first device-side fault in the workspace status word.
DV_DEV void set_status(int *status, int code)
{
    if (status)
        atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------------------
// Storage types.  A 16-byte vector holds EPC elements of T.
template <typename T>
struct Elem;

template <>
struct Elem<float> {
    static constexpr int EPC = 4;
    DV_DEV static void unpack(const uint4 &v, float (&f)[4])
    {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
    DV_DEV static float load(const float *p, size_t i) { return p[i]; }
    DV_DEV static float to_float(float v) { return v; }
    DV_DEV static float from_float(float v) { return v; }
};

template <>
struct Elem<__half> {
    static constexpr int EPC = 8;
    DV_DEV static void unpack(const uint4 &v, float (&f)[8])
    {
        const __half2 *h = reinterpret_cast<const __half2 *>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 t = __half22float2(h[i]);
            f[2 * i] = t.x;
            f[2 * i + 1] = t.y;
        }
    }
    DV_DEV static float load(const __half *p, size_t i) { return __half2float(p[i]); }
    DV_DEV static float to_float(__half v) { return __half2float(v); }
    DV_DEV static __half from_float(float v) { return __float2half_rn(v); }
};

// ---------------------------------------------------------------------------
// Warp and block reductions / scans.
DV_DEV float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

DV_DEV int warp_sum_int(int v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

DV_DEV int warp_incl_scan(int v, int lane)
{
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o)
            v += t;
    }
    return v;
}

// Thread groups that the block-wide helpers below work over.  CtaGroup is
// the whole CTA (__syncthreads).  ConsumerGroup is the first kConsumers
// threads of a CTA whose remaining warp runs on its own (the weight producer
// of the streaming layer kernel): it synchronises on named barrier 1, so the
// other warp never has to join.
struct CtaGroup {
    DV_DEV static int size() { return blockDim.x; }
    DV_DEV static void sync() { __syncthreads(); }
};
constexpr int kConsumers = 384;
struct ConsumerGroup {
    DV_DEV static int size() { return kConsumers; }
    DV_DEV static void sync() { asm volatile("bar.sync 1, 384;" ::: "memory"); }
};

// Exclusive prefix sum over the group (a multiple of 32 threads, <= 1024).
// `scratch` holds >= 33 ints of shared memory.  Returns this thread's
// exclusive prefix; *total receives the group total.  Contains barriers.
template <class Grp = CtaGroup>
DV_DEV int block_excl_scan(int v, int *scratch, int *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nw = Grp::size() >> 5;
    int inc = warp_incl_scan(v, lane);
    if (lane == 31)
        scratch[warp] = inc;
    Grp::sync();
    if (warp == 0) {
        int t = lane < nw ? scratch[lane] : 0;
        int ti = warp_incl_scan(t, lane);
        if (lane < nw)
            scratch[lane] = ti - t;
        if (lane == 31)
            scratch[32] = ti;
    }
    Grp::sync();
    int r = scratch[warp] + inc - v;
    *total = scratch[32];
    Grp::sync();
    return r;
}

// Sum over the group (float); result valid in every thread.  Barriers inside.
template <class Grp = CtaGroup>
DV_DEV float block_sum(float v, float *scratch)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nw = Grp::size() >> 5;
    v = warp_sum(v);
    if (lane == 0)
        scratch[warp] = v;
    Grp::sync();
    if (warp == 0) {
        float t = lane < nw ? scratch[lane] : 0.f;
        t = warp_sum(t);
        if (lane == 0)
            scratch[32] = t;
    }
    Grp::sync();
    float r = scratch[32];
    Grp::sync();
    return r;
}

// ---------------------------------------------------------------------------
// Order-preserving key of a binary32 score: larger float -> larger unsigned.
// -0.0 is folded onto +0.0 so equal scores tie (and the lower index wins).
DV_DEV unsigned score_key(float s)
{
    unsigned u = __float_as_uint(s);
    if (u == 0x80000000u)
        u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Flag hand-off between kernels of one call: the writer publishes its data,
// then stores the flag with release semantics; a reader that sees the flag
// with acquire semantics also sees the data.
DV_DEV int ld_acquire_gpu(const int *p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
DV_DEV void st_release_gpu(int *p, int v)
{
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch (griddepcontrol); no-ops when the kernel was
// launched without the attribute.
DV_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
DV_DEV void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// ---------------------------------------------------------------------------
// How the body of a kernel family waits for its inputs.  Every call site is
// reached by all threads of the CTA.
//
// PdlDep: the body is a kernel of its own, launched as a programmatic
// dependent of the kernel before it.  wait() is the grid dependency, after
// which the body lets its own dependents launch; trigger() lets them launch
// without waiting.
// stamps (optional): this CTA's timeline slots; wait() stamps slot 1.
struct PdlDep {
    unsigned long long *stamps = nullptr;
    DV_DEV void wait() const
    {
        pdl_wait();
        ready();
        pdl_launch_dependents();
    }
    DV_DEV void trigger() const { pdl_launch_dependents(); }
    DV_DEV void ready() const;
};

DV_DEV unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Timeline slot i of a CTA (thread 0; nothing when stamps is NULL).
DV_DEV void chain_stamp(unsigned long long *stamps, int i)
{
    if (stamps && threadIdx.x == 0)
        stamps[i] = global_ns();
}

DV_DEV void PdlDep::ready() const { chain_stamp(stamps, 1); }

// A kernel wrapper's timeline: slot 0 on entry, slot 2 once every thread of
// the CTA has left the body (the barrier only when stamping).
DV_DEV unsigned long long *chain_stamps(unsigned long long *base)
{
    unsigned long long *s =
        (base && blockIdx.y == 0) ? base + (size_t)blockIdx.x * kChainStamps : nullptr;
    chain_stamp(s, 0);
    if (s && threadIdx.x == 0) {
        unsigned sm;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
        s[3] = sm;
    }
    return s;
}
DV_DEV void chain_stamp_end(unsigned long long *s)
{
    if (s) {
        __syncthreads();
        chain_stamp(s, 2);
    }
}

}  // namespace dv
