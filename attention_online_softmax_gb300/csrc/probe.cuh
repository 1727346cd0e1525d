// Measurement aid for the decode time floor ("Tang: a compiler that derives
// GPU kernels and bounds how fast they can run", abstract: a time floor built
// on the traffic bound, the measured launch cost and the DRAM latency).  One
// thread follows a chain of dependent loads through a buffer larger than L2;
// the elapsed global time divided by the number of hops is one DRAM round trip.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace attn {

// An entry that points outside the chain is reported (ATTN_ERR_BOUNDS) and
// ends the walk: out_ns[0] is then 0 and out_ns[1] the bad entry.
__global__ void dram_latency_kernel(const uint32_t* chain, size_t chain_len, int hops, unsigned long long* out_ns) {
  uint32_t idx = 0;
  unsigned long long t0, t1;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (int h = 0; h < hops; ++h) {
    idx = __ldcg(chain + idx);  // L2-only load: no L1 hit on a revisit
    if (idx >= chain_len) {
      report_error(7 /* ATTN_ERR_BOUNDS */, 70, static_cast<int>(idx));
      out_ns[0] = 0;
      out_ns[1] = idx;
      return;
    }
  }
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
  out_ns[0] = t1 - t0;
  out_ns[1] = idx;  // keeps the chain live
}

}  // namespace attn
