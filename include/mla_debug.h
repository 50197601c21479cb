/*
 * mla_debug.h — entry points of the test build of the library
 * (libmla_gb300_debug.so, compiled from the same sources with
 * MLA_DEBUG_CHECKS=1). The release library libmla_gb300.so does not export
 * them. No page has a counterpart: they instrument the decode kernel so tests
 * can see that rarely taken branches ran and that a bounded wait gives up.
 *
 * In the test build the decode kernel also checks every shared-memory
 * address it computes for a plain or cluster store or load (and the tensor
 * memory columns of the P operand) against its own allocation; an address
 * outside it is counted, reported as MLA_ERR_BOUNDS in err_word, and the
 * access is skipped where it is a store the kernel can drop.
 *
 * All calls act on the current device, copy synchronously, and return a
 * cudaError_t value (0 = success).
 */
#ifndef MLA_GB300_DEBUG_H
#define MLA_GB300_DEBUG_H

#ifdef __cplusplus
extern "C" {
#endif

/* Copy the first n (1..4) counters of the decode kernel to host memory:
 *   out[0] warps that rescaled their accumulator in tensor memory because the
 *          running score maximum rose past the lazy-rescale threshold
 *   out[1] shared- or tensor-memory addresses found outside the allocation
 *   out[2], out[3] reserved (0) */
int mla_debug_read_counters(unsigned long long* out, int n);

/* Zero the counters, turn the producer switch off and restore the default
 * wait limit (about 2 s). */
int mla_debug_reset(void);

/* Limit, in SM clock cycles, of every bounded wait in the decode kernel
 * (<= 0 restores the default). */
int mla_debug_set_wait_limit(long long cycles);

/* on != 0: the decode kernel's producer warp loads nothing, so every consumer
 * wait runs into its limit and the call reports MLA_ERR_TIMEOUT in err_word
 * (the results are then not valid). */
int mla_debug_set_skip_producer(int on);

#ifdef __cplusplus
}
#endif
#endif /* MLA_GB300_DEBUG_H */
