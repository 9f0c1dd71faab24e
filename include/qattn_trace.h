/*
 * qattn tracing build -- diagnostics, not part of the library's interface.
 *
 * These functions exist only in the library built with -DQATTN_TRACE
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
 *
 * The same build has a copy probe: the decode kernel's K and V tile copies
 * (the same TMA boxes through the same tensor maps) with nothing consuming
 * them, which times the copy pattern of a decode call on its own.
 */
#ifndef QATTN_TRACE_H_
#define QATTN_TRACE_H_

#include <stdint.h>

#include "qattn.h"

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

/* The copy probe.  On `stream`, one pass over `tiles` ([num_tiles][9]
 * int32, device memory: a KV head, then the cache block of each 16-, 32- or
 * 64-token part of a 128-token tile, -1 where there is none), in the
 * decode's order and split over the SMs as evenly: per tile the K and V
 * boxes of k_cache / v_cache ([num_blocks][Hkv][BS][128], bf16 or, with
 * kv_fp8 = 1, e4m3 codes) into a ring of `stages` tile slots per SM (2 ..
 * 3 for bf16, 2 .. 7 for FP8), a slot reused once its copies have landed;
 * nothing reads them.  Asynchronous; time it with events on `stream`.
 * Block ids outside the cache set QATTN_DEVERR_BLOCK in *err_word (and are
 * skipped), a copy that does not land within 2 s QATTN_DEVERR_TIMEOUT.
 * Returns QATTN_ERR_INVALID_ARG for bad sizes or stage counts. */
int qattn_trace_copy_stream(const void* k_cache, const void* v_cache, int32_t num_blocks,
                            qattn_dims dims, int32_t kv_fp8, const int32_t* tiles,
                            int32_t num_tiles, int32_t stages, int32_t* err_word, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* QATTN_TRACE_H_ */
