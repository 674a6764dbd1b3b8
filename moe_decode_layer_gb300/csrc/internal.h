// Host helpers of api.cu shared with the other host entry points of the library.
#pragma once
#include "../../include/moe_decode.h"
#include "moe_params.h"

namespace moe {
moe_status check_config_host(const moe_decode_config* cfg);
moe_status check_weights_host(const moe_decode_config& cfg, const moe_decode_weights* w);
// Plans the launch shape for a device with `sms` SMs and `smem_optin` bytes of
// opt-in shared memory; fills everything but pointers into scratch and the run's
// rows. ilv: the layout of the slot-interleaved single kernel (MOE_ERR_UNSUPPORTED
// when it does not fit).
moe_status plan_host(const moe_decode_config& cfg, int sms, int smem_optin, Params& p, bool ilv);
// Copies the weight pointers into p.
void bind_weights_host(const moe_decode_weights& w, Params& p);
}  // namespace moe
