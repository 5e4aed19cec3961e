// Device-side status block: the first bytes of every caller workspace.
// Kernels record the first device error (a bounded wait that gave up, a
// failed internal check) here; m2rnn_sync_status reads and clears it.
#pragma once

#include <cstdint>

namespace m2rnn {

struct StatusBlock {
  unsigned int code;    // 0 = ok, else one of kStatus*
  unsigned int detail;  // location code of the first error
  unsigned int pad[62];
};
static_assert(sizeof(StatusBlock) == 256, "status block is 256 bytes");

constexpr unsigned int kStatusTimeout = 1;
constexpr unsigned int kStatusCheck = 2;

// Location codes: kernel id * 100 + site.
constexpr uint32_t kWhereFwdFull = 101, kWhereFwdEmpty = 102, kWhereFwdD = 103,
                   kWhereFwdYFull = 104, kWhereFwdYPeer = 105, kWhereFwdYEmpty = 106,
                   kWhereFwdDrain = 107, kWhereFwdExit = 108,
                   kWhereFwdH = 109;
constexpr uint32_t kWhereBwdFull = 201, kWhereBwdCEmpty = 202, kWhereBwdTReady = 203,
                   kWhereBwdTFree = 204, kWhereBwdXFull = 205, kWhereBwdXEmpty = 206,
                   kWhereBwdDrain = 207, kWhereBwdDW = 208, kWhereBwdZFull = 209;
// Input checks: an entry of W outside the fp16 range (|W| >= 65520) that the
// fp16 state-operand kernels cannot represent.
constexpr uint32_t kWhereWRange = 301;
// An entry of q with |q| >= 65536 (or not finite) in a forward whose readout
// takes q as an fp16 operand (the V = 64 and V = 16 warp-MMA forwards with
// readout warps).
constexpr uint32_t kWhereQRange = 302;

__device__ __forceinline__ void report_device_error(StatusBlock* s, unsigned int code,
                                                    uint32_t where) {
  if (s != nullptr && atomicCAS(&s->code, 0u, code) == 0u) atomicExch(&s->detail, where);
}

}  // namespace m2rnn
