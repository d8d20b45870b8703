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

#ifdef __cplusplus
}
#endif

#endif /* GDN_TESTING_H */
