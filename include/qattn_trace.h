/*
 * qattn tracing build -- diagnostics, not part of the library's interface.
 *
 * These three functions exist only in the library built with -DQATTN_TRACE
 * (paged_kv_gqa_07_gb300/build.py, build(trace=True), which writes
 * _build/trace/libqattn_trace.so).  In that build the decode kernel and the
 * split-KV merge kernel record a %globaltimer stamp (nanoseconds) per CTA at
 * their phase boundaries; the kernels are otherwise the same code as in the
 * regular library.  Stamps of CTAs beyond the buffers' capacity are dropped.
 *
 * Decode kernel, per CTA (slots; unused slots stay 0):
 *   0 entry, 1 plan done, 2 first scores read by the softmax,
 *   3 every copy issued by the producer, 4 softmax done, 5 CTA done.
 * Merge kernel, per CTA: 0 entry, 1 the decode grid's completion seen, 2 done.
 *
 * The buffers keep the last launch's stamps (a later launch overwrites the
 * slots of the CTAs it runs); clear them before the launch to read.
 */
#ifndef QATTN_TRACE_H_
#define QATTN_TRACE_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Capacities: decode CTAs recorded, slots per decode CTA, merge CTAs
 * recorded.  Host pointers; returns QATTN_OK. */
int qattn_trace_dims(int32_t* decode_ctas, int32_t* decode_slots, int32_t* merge_ctas);

/* Zero both stamp buffers on the current device (synchronous). */
int qattn_trace_clear(void);

/* Copy the stamp buffers of the current device to host memory (synchronous):
 * decode_host [decode_ctas * decode_slots], merge_host [merge_ctas * 4]. */
int qattn_trace_read(uint64_t* decode_host, uint64_t* merge_host);

#ifdef __cplusplus
}
#endif

#endif /* QATTN_TRACE_H_ */
