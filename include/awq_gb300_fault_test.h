/*
 * awq_gb300_fault_test.h -- test-only entry point of the fault-test build of
 * the library (libawq_gb300_fault_test.so, compiled with AWQ_FAULT_TEST). The
 * regular library does not export it. The pages have no counterpart of this
 * call: it exists so that the bounded waits of the kernels can be made to run
 * out on purpose, without a GPU fault, and the library's recovery checked.
 *
 * In the fault-test build every device-side wait gives up after about 4e6 SM
 * clock cycles (about 2 ms) instead of 4e9, and:
 *
 * awq_test_inject_fault(on) -- while `on` is non-zero, every decode and
 *   prefill kernel launched afterwards (awq_linear_forward and the calls built
 *   on it) has the TMA producer of its CTA 0 issue no copy. That CTA's
 *   consumer warps then wait on a stage barrier that never fills; the waits
 *   run out, record AWQ_ERR_TIMEOUT in the device status word, and the
 *   kernel returns. Other CTAs that wait for CTA 0's partial sums give up the
 *   same way. Nothing traps, faults or spins without a limit. The result of
 *   such a call is not defined; awq_last_device_status() then returns
 *   AWQ_ERR_TIMEOUT and resets the split-K counters. Host-side switch; takes
 *   effect at the next launch. No CUDA call.
 */
#ifndef AWQ_GB300_FAULT_TEST_H
#define AWQ_GB300_FAULT_TEST_H

#ifdef __cplusplus
extern "C" {
#endif

void awq_test_inject_fault(int on);

#ifdef __cplusplus
}
#endif

#endif /* AWQ_GB300_FAULT_TEST_H */
