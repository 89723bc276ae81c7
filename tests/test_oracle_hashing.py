"""Pins for the oracle's block digests (CPU only): the published test vectors
of the primitives it builds on (RFC 7693 BLAKE2b, FIPS 180-4 SHA-256, RFC 4231
HMAC-SHA256, the BLAKE2 keyed known-answer test), and the properties the two
digests exist for."""
import hashlib
import hmac

import numpy as np

from oracle import hashing


def test_primitives_published_vectors():
    assert hashlib.blake2b(b"abc").hexdigest() == (
        "ba80a53f981c4d0d6a2797b69f12f6e94c212f14685ac4b74b12bb6fdbffa2d1"
        "7d87c5392aab792dc252d5de4533cc9518d38aa8dbf1925ab92386edd4009923")
    assert hashlib.blake2b(b"", key=bytes(range(64))).hexdigest() == (
        "10ebb67700b1868efb4417987acf4690ae9d972fb7a590c2f02871799aaa4786"
        "b5e996e8f0f4eb981fc214b005f42d2ff4233499391653df7aefcbc13fc51568")
    assert hashlib.sha256(b"abc").hexdigest() == (
        "ba7816bf8f01cfea414140de5dae2223b00361a396177a9cb410ff61f20015ad")
    assert hmac.new(b"Jefe", b"what do ya want for nothing?", hashlib.sha256).hexdigest() == (
        "5bdcc146bf60754e6a042426089575c75a003f089d2739839dec58b964ec3843")


def test_tenant_keys():
    m = b"master secret"
    assert hashing.tenant_key(m, "acme") != hashing.tenant_key(m, "globex")
    assert hashing.tenant_key(m, None) == hashing.tenant_key(m, "")       # public namespace
    assert hashing.tenant_key(m, "acme") == hmac.new(m, b"hc-tenant:acme", hashlib.sha256).digest()
    assert len(hashing.tenant_key(m, "acme")) == 32


def test_digest_properties():
    r = np.random.default_rng(0)
    key = hashing.tenant_key(b"m", "acme")
    a = r.integers(0, 150000, 16 * 5 + 7)
    p, c = hashing.block_digests(a, 16, key)
    assert p.shape == (6, 16) and c.shape == (6, 16)
    # block 0: the prefix digest is the content digest (nothing before it)
    assert np.array_equal(p[0], c[0])
    # swap blocks 1 and 2: contents follow the tokens, prefixes change from block 1 on
    b = a.copy()
    b[16:32], b[32:48] = a[32:48], a[16:32]
    p2, c2 = hashing.block_digests(b, 16, key)
    assert np.array_equal(c2[1], c[2]) and np.array_equal(c2[2], c[1])
    assert np.array_equal(p2[0], p[0]) and not np.array_equal(p2[1], p[1])
    assert not np.array_equal(p2[3], p[3])          # the chain carries the change
    # another tenant's key gives unrelated digests
    p3, c3 = hashing.block_digests(a, 16, hashing.tenant_key(b"m", "globex"))
    assert not np.any(np.all(c3 == c, axis=1))
    # a definition spot check: block 1's prefix digest
    want = hashlib.blake2b(p[0].tobytes() + a[16:32].astype("<i4").tobytes(), digest_size=16, key=key)
    assert p[1].tobytes() == want.digest()
