/*
 * gq_testing.h -- fault injection for the failure-detection tests of libgq.so.
 *
 * Not part of the data path.  The pages describe a watchdog that times out a stuck
 * collective and reports it ("torch_npu distributed module" article, hwcomputing.csdn.net,
 * §5 Watchdog runLoop: poll, detect timeout, dump and raise).  Here every device-side wait is
 * bounded; this hook lets a test make one run out without faulting anything.
 */
#ifndef GQ_TESTING_H
#define GQ_TESTING_H

#include <stdint.h>

#include "gq.h"

#ifdef __cplusplus
extern "C" {
#endif

/* On the current device, make every later gq_fused_allreduce_sim bulk-copy wait expect
 * `extra_bytes` more than its copies deliver (so the wait cannot complete) and give up after
 * `limit_ns`; the kernel then records GQ_ERR_TIMEOUT, finishes its work on what did arrive,
 * waits once more (bounded) and returns.  gq_testing_inject_copy_stall(0, 0) restores the
 * defaults (no extra bytes, 2 s limit).  Synchronous; returns GQ_ERR_CUDA if the update of the
 * device settings failed. */
gq_status gq_testing_inject_copy_stall(uint32_t extra_bytes, uint64_t limit_ns);

#ifdef __cplusplus
}
#endif
#endif /* GQ_TESTING_H */
