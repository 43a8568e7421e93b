/*
 * wkv7_debug.h - extra entry points of the debug build of the WKV7 library
 * (libwkv7_debug.so, compiled with WKV7_DEBUG). The product library does not
 * export them. They have no counterpart on the pages: they exist to test the
 * library's own error paths, WKV7_ERR_TIMEOUT and WKV7_ERR_BOUNDS.
 *
 * Every wait of a kernel on an mbarrier is bounded: after the limit it sets
 * the device status word, drains the copy it was waiting for and leaves the
 * kernel, and wkv7_status() then returns WKV7_ERR_TIMEOUT and clears the
 * word. In the debug build the limit is 1 ms instead of about 2 s.
 *
 * In the debug build every plain (non-TMA) global load and store of the scan
 * kernels (forward, backward, checkpointing forward, every chunked form)
 * checks its address against the buffer it belongs to, as the library sized
 * it from B, T, H, N and the checkpoint interval. An access outside it is
 * skipped (a load reads zero) and sets the status word, and wkv7_status()
 * then returns WKV7_ERR_BOUNDS.
 */
#ifndef WKV7_DEBUG_H
#define WKV7_DEBUG_H

#include <stddef.h>

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

/* From now on the kernels check their accesses against buffers `bytes`
 * shorter than they are (each buffer's last `bytes` bytes count as outside
 * it), so the checks skip the stores and loads there and wkv7_status() returns
 * WKV7_ERR_BOUNDS; no access ever leaves the real buffer. bytes = 0 restores
 * normal operation. For the test of the checks themselves. Process-wide;
 * returns WKV7_OK. */
int wkv7_debug_cut_extents(size_t bytes);

#ifdef __cplusplus
}
#endif

#endif /* WKV7_DEBUG_H */
