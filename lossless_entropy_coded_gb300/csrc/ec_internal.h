/*
 * ec_internal.h -- host descriptor of an encoded matrix, shared by the host codec
 * (ec_host.cpp) and the kernel launchers (ec_kernels.cu).
 */
#ifndef EC_INTERNAL_H_
#define EC_INTERNAL_H_

#include <stdint.h>

#include "../../include/ec.h"
#include "ec_format.h"

struct ec_matrix {
    int32_t kind;
    int32_t device;
    ec_blob_header hdr;        /* host copy of the device header */
    uint8_t* d_blob;           /* device blob (owned); NULL for a host-only matrix */
    uint8_t* h_blob;           /* host copy, kept only when device < 0 */
    /* host-side statistics */
    uint8_t lengths[256];
    uint64_t counts[256];      /* exponent (Huffman) or rANS symbol histogram, padding included */
    uint32_t freqs[256];       /* rANS */
    int64_t payload_bits, raw_bytes, aux_bytes, table_bytes;
    double entropy;
};

/* Device status word (one per device, allocated on first use). */
int ec_internal_status_ptr(int device, int** out);

#endif
