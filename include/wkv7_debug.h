/*
 * wkv7_debug.h - extra entry point of the debug build of the WKV7 library
 * (libwkv7_debug.so, compiled with WKV7_DEBUG). The product library does not
 * export it. It has no counterpart on the pages: it exists to test the
 * library's own error path, WKV7_ERR_TIMEOUT.
 *
 * Every wait of a kernel on an mbarrier is bounded: after the limit it sets
 * the device status word, drains the copy it was waiting for and leaves the
 * kernel, and wkv7_status() then returns WKV7_ERR_TIMEOUT and clears the
 * word. In the debug build the limit is 1 ms instead of about 2 s.
 */
#ifndef WKV7_DEBUG_H
#define WKV7_DEBUG_H

#ifdef __cplusplus
extern "C" {
#endif

/* on != 0: from now on, the scalar forward kernel (fp32 inputs, or N other
 * than 64) issues no load, and no expected byte count, for the last chunk of
 * every head, so every CTA's wait for that chunk runs out after 1 ms with no
 * copy in flight; the forward call itself returns WKV7_OK and the next
 * wkv7_status() returns WKV7_ERR_TIMEOUT. on = 0 restores normal operation.
 * Process-wide; returns WKV7_OK. */
int wkv7_debug_skip_last_load(int on);

/* which = 1: the split backward's per-chunk output pass runs the kernel whose
 * products are tcgen05.mma on tensor memory (persistent, four CTAs per SM)
 * instead of the default one on warp-level mma.sync products (which = 0); the
 * results agree to rounding. For side-by-side timing and parity; the product
 * library always runs the default. Process-wide; returns WKV7_OK. */
int wkv7_debug_out_kernel(int which);

#ifdef __cplusplus
}
#endif

#endif /* WKV7_DEBUG_H */
