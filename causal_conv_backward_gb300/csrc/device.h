// device.h - what the host side asks of the device: the calling thread's
// current context, by its unique id, and the SM count the plans assume.
//
// Per-device state the library caches on the host (kernel attributes, the
// no-allocation scratch address) belongs to one context: a device reset
// (cudaDeviceReset, or a framework that releases and re-creates the primary
// context) starts a new one with none of it. Keying such caches on the
// context's id makes the first call in a new context set them up again.
#pragma once

#include <stdint.h>

namespace mcc1d {

// Unique id of the calling thread's current context (never reused within a
// process), or 0 when no context is current or the driver cannot say.
unsigned long long current_context_id();

// The plans cut every problem into kNumSMs x (CTAs per SM) persistent CTAs,
// a function of the shape alone so that results never depend on the device.
// On a device (or partition) with fewer SMs part of that grid would run as a
// second wave at about twice the time. Returns kOk when the current device
// has at least kNumSMs SMs, kErrDevice when it has fewer, kErrCuda when the
// runtime cannot say. The count is read once per device.
int32_t check_current_device();
// The check itself, for a given SM count.
int32_t check_sm_count(int32_t sm_count);
// SM count of the current device (cached per device), or 0 when unknown.
int32_t current_device_sm_count();

}  // namespace mcc1d
