// Host-side argument checks of the C-ABI entry points (defined in api.cu).  Each
// returns IPTTT_OK or the status the entry point hands back unchanged.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "ipttt.h"

namespace ipttt {

// dims: non-null, a known dtype, 1 <= d, d_ff <= 2^20, batch >= 0 (need_batch), w0_per_seq 0 or 1,
// bf16 mode: d and d_ff multiples of 8.  IPTTT_ERR_INVALID_ARG otherwise.
ipttt_status check_dims(const ipttt_dims* dims, bool need_batch);
// L >= 0 a multiple of B >= 1 (bf16 mode: B a multiple of 16), token and weight rows within int32.
ipttt_status check_chunking(const ipttt_dims* dims, int64_t L, int64_t B);
// The current device has compute capability 10.3 (IPTTT_ERR_UNSUPPORTED otherwise).
ipttt_status check_device();
// Every pointer non-null and 16-byte aligned (checked first, without a CUDA call), then the
// device, then every pointer device or managed memory.
ipttt_status check_ptr_list(const void* const* ps, int n);
template <size_t N>
ipttt_status check_ptrs(const void* const (&ps)[N]) {
  return check_ptr_list(ps, static_cast<int>(N));
}

}  // namespace ipttt
