"""Host-side behaviour of the photo store (kda_photo_*) that needs no GPU: the
capacity rule (a directory alone means 2 photos, a given capacity always wins, 0 is
off), the directory check, lookups in an empty store, and argument errors returned
before any device work."""
import ctypes

import pytest

import linear_attention_mixer_gb300 as K


@pytest.fixture(scope="module", autouse=True)
def _built():
    from linear_attention_mixer_gb300 import build
    build.build()


def test_capacity_rule(tmp_path):
    cases = [(-1, None, 0), (-1, str(tmp_path), 2), (0, str(tmp_path), 0), (5, None, 5), (1, str(tmp_path), 1)]
    for cap, d, want in cases:
        ps = K.kda_photo_store_create(cap, d)
        try:
            assert K.kda_photo_capacity(ps) == want, (cap, d)
            assert K.kda_photo_count(ps) == 0
        finally:
            K.kda_photo_store_free(ps)
    assert K.kda_photo_capacity(None) == 0 and K.kda_photo_count(None) == 0
    K.kda_photo_store_free(None)


def test_directory_must_exist(tmp_path):
    with pytest.raises(K.KdaError) as e:
        K.kda_photo_store_create(2, str(tmp_path / "missing"))
    assert e.value.status == K.KDA_ERR_INVALID
    f = tmp_path / "a_file"
    f.write_text("x")
    with pytest.raises(K.KdaError) as e:
        K.kda_photo_store_create(2, str(f))
    assert e.value.status == K.KDA_ERR_INVALID


def test_find_in_empty_store_and_argument_errors():
    L = K.lib()
    ps = K.kda_photo_store_create(3)
    try:
        assert K.kda_photo_find(ps, [1, 2, 3]) == (-1, 0)
        assert K.kda_photo_find(ps, []) == (-1, 0)
        pid, plen = ctypes.c_int32(), ctypes.c_int64()
        assert L.kda_photo_find(ps, None, -1, ctypes.byref(pid), ctypes.byref(plen)) == K.KDA_ERR_INVALID
        assert L.kda_photo_find(ps, None, 4, ctypes.byref(pid), ctypes.byref(plen)) == K.KDA_ERR_INVALID
        assert L.kda_photo_find(None, None, 0, ctypes.byref(pid), ctypes.byref(plen)) == K.KDA_ERR_INVALID
        # take / restore reject their arguments before touching a device
        assert L.kda_photo_take(ps, None, 1, 0, None, 0, None, None) == K.KDA_ERR_INVALID
        arr = (ctypes.c_void_p * 1)(None)
        assert L.kda_photo_take(ps, arr, 1, 0, None, 0, None, None) == K.KDA_ERR_INVALID
        assert L.kda_photo_take(ps, arr, 0, 0, None, 0, None, None) == K.KDA_ERR_INVALID
        assert L.kda_photo_take(None, arr, 1, 0, None, 0, None, None) == K.KDA_ERR_INVALID
        assert L.kda_photo_restore(ps, 0, None, 1, 0, None) == K.KDA_ERR_INVALID
        assert L.kda_photo_restore(None, 0, arr, 1, 0, None) == K.KDA_ERR_INVALID
        assert "NULL" in K.kda_last_error()
        assert L.kda_photo_store_create(2, None, None) == K.KDA_ERR_INVALID
    finally:
        K.kda_photo_store_free(ps)
