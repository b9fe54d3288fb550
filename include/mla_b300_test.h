/*
 * mla_b300_test.h -- test-only entry point of the library's test build.
 *
 * Only libmla_b300_testhooks.so exports this symbol: the same sources
 * compiled with MLA_TEST_HOOKS, where the tensor-core decode kernel's
 * bounded waits give up after 20 ms instead of 2 s. The shipped
 * libmla_b300.so has neither. There is no counterpart in the method: this
 * exists so that a test can make a device-side wait run out without any
 * fault.
 */
#ifndef MLA_B300_TEST_H
#define MLA_B300_TEST_H

#ifdef __cplusplus
extern "C" {
#endif

/* on != 0: every following mla_decode_attn launch on the tensor-core path
 * issues no page copies, so its waits for page data run out; the kernel
 * then sets MLA_DEV_TIMEOUT in the status word, drains what it issued and
 * returns. on == 0 restores normal launches. Host state only; not thread
 * safe. */
void mla_test_withhold_pages(int on);

#ifdef __cplusplus
}
#endif
#endif /* MLA_B300_TEST_H */
