/*
 * gdn_testing.h -- test hooks of libgdn. Not part of the stable interface:
 * they exist so that tests can reach code paths that ordinary inputs never
 * take.
 */
#ifndef GDN_TESTING_H
#define GDN_TESTING_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Limit, in nanoseconds of the GPU's global timer, of the first bounded wait
 * of the prefill's sequential pass and of each CTA's first tile-copy wait in
 * the multi-token conv, for every later call in this process (0 restores the
 * default of 2 s). A tiny value makes those waits give up while the work they
 * wait for is still in flight, so a test can check that the kernels then set
 * their bit of the device error word (gdn_check_device), drain what they
 * issued and return, and that the next call runs normally. Every other wait
 * keeps the default limit.
 */
void gdn_testing_set_first_wait_ns(uint64_t ns);

/*
 * The row slices per V head that the launchers choose for n_seq sequences of
 * n_v_heads V heads, r = n_v_heads / n_qk_heads, on a device with sms SMs:
 * *decode_split for the single-token decode step, *scan_split for the
 * token-serial scans (gdn_layer_scan, gdn_recurrence_scan); the verify steps use
 * *decode_split too. Host-only: no device is touched, so the choice can be
 * tested for any SM count.
 */
void gdn_testing_row_splits(int32_t n_seq, int32_t n_v_heads, int32_t r, int32_t sms,
                            int32_t *decode_split, int32_t *scan_split);

#ifdef __cplusplus
}
#endif

#endif /* GDN_TESTING_H */
