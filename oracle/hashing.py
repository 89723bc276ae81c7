"""Block digests for cache lookup, keyed per tenant.

ORACLE (test infrastructure only; see the package docstring).

The page computes "two deterministic 128-bit BLAKE2b digests per token block
(default 16 or 64 tokens)", all keyed "by a per-tenant secret derived via
HMAC-SHA256", with an explicit "public" namespace for shared system prompts
["HyperCache - Distributed KV-cache quantization and relative RoPE reuse",
"Core Design", item 1 "Dual-Mode Block Hashing"].  The list naming the two
digests is lost from the page, and so is the key derivation; the reading taken
(the plainest one that serves both kinds of reuse the page describes - exact
causal prefixes, and chunks reused at a new offset with the relative RoPE):

* tenant secret: K = HMAC-SHA256(master, b"hc-tenant:" + tenant), 32 bytes;
  the public namespace uses K = HMAC-SHA256(master, b"hc-public");
* block j holds tokens [j*B, (j+1)*B) (the last block may be short), as
  little-endian int32;
* prefix digest  p_j = BLAKE2b-128(key K; p_{j-1} || tokens of block j), with
  p_{-1} the empty string: it names the block together with everything
  before it (exact prefix reuse);
* content digest c_j = BLAKE2b-128(key K; tokens of block j): it names the
  block's tokens wherever they sit (chunk reuse at a new offset).

hashlib and hmac (the standard library's implementations of RFC 7693 and
RFC 2104 / FIPS 180-4) are the steps.
"""
import hashlib
import hmac

import numpy as np

DIGEST_BYTES = 16


def tenant_key(master, tenant=None):
    msg = b"hc-public" if not tenant else b"hc-tenant:" + tenant.encode()
    return hmac.new(bytes(master), msg, hashlib.sha256).digest()


def block_digests(tokens, block_size, key):
    """(prefix [n_blocks, 16] uint8, content [n_blocks, 16] uint8)."""
    t = np.asarray(tokens, dtype="<i4")
    n_blocks = -(-len(t) // block_size)
    prefix = np.zeros((n_blocks, DIGEST_BYTES), np.uint8)
    content = np.zeros((n_blocks, DIGEST_BYTES), np.uint8)
    prev = b""
    for j in range(n_blocks):
        blk = t[j * block_size:(j + 1) * block_size].tobytes()
        c = hashlib.blake2b(blk, digest_size=DIGEST_BYTES, key=key).digest()
        p = hashlib.blake2b(prev + blk, digest_size=DIGEST_BYTES, key=key).digest()
        content[j] = np.frombuffer(c, np.uint8)
        prefix[j] = np.frombuffer(p, np.uint8)
        prev = p
    return prefix, content
