// Links between the host-side objects of libpagedattn.so (not part of the C ABI).
#pragma once

#include "../../include/pa.h"

namespace pa {

// A prefix cache holds block references on its allocator: the allocator stays
// allocated while caches are attached, even after pa_allocator_destroy, and is
// released when the last of them detaches.  Destruction order is then free.
void allocator_attach(pa_allocator* a);
void allocator_detach(pa_allocator* a);

}  // namespace pa
