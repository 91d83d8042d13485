// fr_trace.cuh -- timeline instrumentation of the decode attention kernels
// (compile-time option, off in the library). With FR_TRACE defined, CTA b
// (b = blockIdx.y * gridDim.x + blockIdx.x, b < 1024) of an attention kernel
// writes global-timer stamps into 64 slots at workspace + FR_TRACE_OFFSET +
// 512 b (the kernel's argument struct is `a`, its status word the start of
// the workspace); slot 63 holds the SM the CTA ran on. The merge kernel's CTA
// b < 1024 stamps slots 1024 + b the same way (FR_STAMP_AT, given the
// workspace start). gqa_kv_head_gb300.trace builds that variant into its own
// library and prints the timeline.
#pragma once

#ifdef FR_TRACE
#ifndef FR_TRACE_OFFSET
#define FR_TRACE_OFFSET (32u << 20)
#endif
#define FR_TRACE_CTA() (blockIdx.y * gridDim.x + blockIdx.x)
#define FR_TRACE_AT(ws, slot)                                                                               \
    (reinterpret_cast<unsigned long long*>(reinterpret_cast<unsigned char*>(ws) + FR_TRACE_OFFSET)[slot])
#define FR_STAMP(i)                                                                                         \
    do {                                                                                                    \
        if (FR_TRACE_CTA() < 1024u) FR_TRACE_AT(a.status, FR_TRACE_CTA() * 64 + (i)) = global_ns();         \
    } while (0)
#define FR_STAMP_SMID()                                                                                     \
    do {                                                                                                    \
        unsigned smid_;                                                                                     \
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid_));                                                  \
        if (FR_TRACE_CTA() < 1024u) FR_TRACE_AT(a.status, FR_TRACE_CTA() * 64 + 63) = smid_;                \
    } while (0)
#define FR_STAMP_AT(ws, i)                                                                                  \
    do {                                                                                                    \
        if (blockIdx.x < 1024u) FR_TRACE_AT(ws, (1024u + blockIdx.x) * 64 + (i)) = global_ns();             \
    } while (0)
#define FR_STAMP_SMID_AT(ws)                                                                                \
    do {                                                                                                    \
        unsigned smid_;                                                                                     \
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid_));                                                  \
        if (blockIdx.x < 1024u) FR_TRACE_AT(ws, (1024u + blockIdx.x) * 64 + 63) = smid_;                    \
    } while (0)
#else
#define FR_STAMP(i) \
    do {            \
    } while (0)
#define FR_STAMP_SMID() \
    do {                \
    } while (0)
#define FR_STAMP_AT(ws, i) \
    do {                   \
        (void)(ws);        \
    } while (0)
#define FR_STAMP_SMID_AT(ws) \
    do {                     \
        (void)(ws);          \
    } while (0)
#endif
