// xp_trace.cuh -- optional per-CTA timeline stamps (a development aid).
//
// Compiled out entirely unless the library is built with -DXP_TRACE.  In a
// trace build every kernel that uses XP_TRACE_MARK(slot) records the global
// timer (ns) of the moment one of its threads reached `slot` into a per
// translation unit array of kTraceCtas x kTraceSlots stamps (CTA-major), and
// slot kTraceSlots-1 of each CTA holds the SM it ran on.  The translation
// unit exports a reader (XP_TRACE_READER) that copies the array to the host
// and clears it.  Stamps are plain stores: a slot that several kernels of one
// launch sequence share keeps the last writer.
#pragma once

#ifdef XP_TRACE
#include <cuda_runtime.h>
#include <stdint.h>

namespace xp {
constexpr int kTraceCtas = 1024;
constexpr int kTraceSlots = 64;
static __device__ unsigned long long g_trace[kTraceCtas * kTraceSlots];

__device__ __forceinline__ void trace_mark(int slot) {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  const unsigned int b = blockIdx.x;
  if (b < (unsigned)kTraceCtas) {
    g_trace[b * kTraceSlots + slot] = t;
    unsigned int sm;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
    g_trace[b * kTraceSlots + kTraceSlots - 1] = sm;
  }
}
}  // namespace xp

#define XP_TRACE_MARK(slot) ::xp::trace_mark(slot)
// record the SM this CTA runs on in `slot` (instead of a time)
#define XP_TRACE_SM(slot)                                                              \
  do {                                                                                 \
    unsigned int sm_;                                                                  \
    asm volatile("mov.u32 %0, %%smid;" : "=r"(sm_));                                   \
    if (blockIdx.x < (unsigned)::xp::kTraceCtas) ::xp::g_trace[blockIdx.x * ::xp::kTraceSlots + (slot)] = sm_ + 1; \
  } while (0)
// extern "C" int name(void* host, size_t bytes): copy the stamps out, then zero them
#define XP_TRACE_READER(name)                                                              \
  extern "C" __attribute__((visibility("default"))) int name(void* host, size_t bytes) {   \
    if (bytes > sizeof(::xp::g_trace)) bytes = sizeof(::xp::g_trace);                      \
    if (cudaMemcpyFromSymbol(host, ::xp::g_trace, bytes) != cudaSuccess) return -1;        \
    static unsigned long long zero[::xp::kTraceCtas * ::xp::kTraceSlots];                  \
    return cudaMemcpyToSymbol(::xp::g_trace, zero, sizeof(zero)) == cudaSuccess ? 0 : -1;  \
  }
#else
#define XP_TRACE_MARK(slot) ((void)0)
#define XP_TRACE_SM(slot) ((void)0)
#define XP_TRACE_READER(name)
#endif
