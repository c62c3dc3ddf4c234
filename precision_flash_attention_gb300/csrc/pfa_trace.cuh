// Optional phase timestamps for one CTA, compiled only into a development
// build (-DPFA_TRACE); in the product build every macro here is empty.
//
// Each trace slot is written by exactly one thread, which keeps its own count
// in a register: an event costs one clock read and one fire-and-forget store,
// so the traced schedule stays close to the untraced one. Word layout: event
// id in bits 56-63, iteration in bits 40-55, SM clock in bits 0-39. The host
// zeroes the buffer before the traced launch; unused words stay zero.
#pragma once

#ifdef PFA_TRACE
// The buffer comes with a host reader `<name>_read(out, clear)`: clear != 0
// zeroes the buffer, otherwise its 8 x 1024 words are copied to `out`.
#define PFA_TRACE_BUFFER(name)                                                                \
  __device__ unsigned long long name[8][1024];                                                 \
  extern "C" int name##_read(unsigned long long* out, int clear) {                             \
    void* p_ = nullptr;                                                                        \
    cudaDeviceSynchronize();                                                                   \
    if (cudaGetSymbolAddress(&p_, name) != cudaSuccess) return -1;                             \
    if (clear) return cudaMemset(p_, 0, sizeof(name)) == cudaSuccess ? 0 : -1;                 \
    return cudaMemcpy(out, p_, sizeof(name), cudaMemcpyDeviceToHost) == cudaSuccess ? 0 : -1;  \
  }                                                                                            \
  static_assert(true, "")
#define PFA_TRACE_DECL() unsigned int pfa_trace_n_ = 0
#define PFA_TRACE_EVENT(buf, slot, ev, j)                                                      \
  do {                                                                                         \
    if (blockIdx.x == PFA_TRACE_BLOCK) {                                                       \
      const unsigned long long c_ = clock64();                                                 \
      if (pfa_trace_n_ < 1024)                                                                 \
        buf[slot][pfa_trace_n_] = (static_cast<unsigned long long>(ev) << 56) |                \
                                  (static_cast<unsigned long long>((j) & 0xFFFF) << 40) |      \
                                  (c_ & 0xFFFFFFFFFFull);                                      \
      ++pfa_trace_n_;                                                                          \
    }                                                                                          \
  } while (0)
#else
#define PFA_TRACE_BUFFER(name) static_assert(true, "")
#define PFA_TRACE_DECL() static_assert(true, "")
#define PFA_TRACE_EVENT(buf, slot, ev, j) \
  do {                                    \
  } while (0)
#endif
