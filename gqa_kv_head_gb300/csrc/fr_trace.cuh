// fr_trace.cuh -- timeline instrumentation of the keys-on-M decode attention
// kernel (compile-time option, off in the library). With FR_TRACE defined,
// CTA b writes global-timer stamps into 64 slots at workspace +
// FR_TRACE_OFFSET + 512 b (the kernel's argument struct is `a`, its status
// word the start of the workspace); slot 63 holds the SM the CTA ran on.
// gqa_kv_head_gb300.trace builds that variant into its own library and prints
// the timeline.
#pragma once

#ifdef FR_TRACE
#ifndef FR_TRACE_OFFSET
#define FR_TRACE_OFFSET (32u << 20)
#endif
#define FR_TRACE_SLOTS()                                                                                    \
    reinterpret_cast<unsigned long long*>(reinterpret_cast<unsigned char*>(a.status) + FR_TRACE_OFFSET)
#define FR_STAMP(i)                                                                                         \
    do {                                                                                                    \
        FR_TRACE_SLOTS()[blockIdx.x * 64 + (i)] = global_ns();                                              \
    } while (0)
#define FR_STAMP_SMID()                                                                                     \
    do {                                                                                                    \
        unsigned smid_;                                                                                     \
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid_));                                                  \
        FR_TRACE_SLOTS()[blockIdx.x * 64 + 63] = smid_;                                                     \
    } while (0)
#else
#define FR_STAMP(i) \
    do {            \
    } while (0)
#define FR_STAMP_SMID() \
    do {                \
    } while (0)
#endif
