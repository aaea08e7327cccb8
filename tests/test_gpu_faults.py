"""Host-side fault injection at the boundary; no GPU fault is provoked. A snapshot
blob with any header field corrupted is refused with KDA_ERR_BLOB before a byte is
copied, for host and device blobs alike, and the state is left as it was. A state far
beyond the device's memory is refused with KDA_ERR_OOM without leaking. The library
keeps working after each refusal."""
import numpy as np
import pytest
import torch

import kda_inputs as KI
import linear_attention_mixer_gb300 as K
from tests.kda_testutil import download_state, upload_state

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from linear_attention_mixer_gb300 import build
    build.build()
    torch.cuda.set_device(0)


def _corruptions():
    """(field, value) pairs, each of which makes a one-slot FP32 H=2 d=128 blob invalid."""
    sb, tb = 2 * 128 * 128 * 4, 3 * 3 * 2 * 128 * 4
    return [("magic", 0x12345678), ("version", K.KDA_BLOB_VERSION + 1), ("num_heads", 3), ("head_dim", 64),
            ("conv_kernel", 3), ("io_dtype", K.KDA_BF16), ("n_slots", 2), ("state_bytes_per_slot", sb + 4),
            ("tail_bytes_per_slot", tb + 4)]


@pytest.mark.parametrize("on_device", [False, True])
def test_corrupted_blob_is_refused_and_the_state_untouched(on_device):
    H, d = 2, 128
    cfg = K.kda_config(H, d, K.KDA_F32)
    st = K.kda_state_alloc(cfg, 2)
    try:
        upload_state(cfg, st, [0, 1], KI.make_state(2, H, d, 5), KI.make_tail(2, H, d, 4, 5, bf16=False))
        before = download_state(cfg, st, [0, 1])
        good = torch.empty(K.kda_state_blob_bytes(st, 1), dtype=torch.uint8)
        K.kda_state_snapshot(st, [0], good)
        torch.cuda.synchronize()
        for field, value in _corruptions():
            hdr = K.kda_blob_header.from_buffer_copy(bytes(good[:64].numpy()))
            setattr(hdr, field, value)
            bad = torch.cat([torch.frombuffer(bytearray(bytes(hdr)), dtype=torch.uint8), good[64:]])
            if on_device:
                bad = bad.cuda()
            with pytest.raises(K.KdaError) as e:
                K.kda_state_restore(st, [1], bad)
            assert e.value.status == K.KDA_ERR_BLOB, field
        torch.cuda.synchronize()
        after = download_state(cfg, st, [0, 1])
        assert np.array_equal(before[0], after[0]) and np.array_equal(before[1], after[1])
        # the intact blob still goes back, into the other slot
        K.kda_state_restore(st, [1], good.cuda() if on_device else good)
        S, t = download_state(cfg, st, [0, 1])
        assert np.array_equal(S[1], S[0]) and np.array_equal(t[1], t[0])
        assert K.kda_state_poll_error(st) == 0
    finally:
        K.kda_state_free(st)


def test_state_beyond_device_memory_is_refused_without_leaking():
    cfg = K.kda_config(96, 128, K.KDA_BF16)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    # one million slots of 6.3 MB: several TB, which the driver refuses outright
    with pytest.raises(K.KdaError) as e:
        K.kda_state_alloc(cfg, 1_000_000)
    assert e.value.status == K.KDA_ERR_OOM
    assert torch.cuda.mem_get_info()[0] >= free0 - (64 << 20)
    # the library and the device are fine afterwards
    st = K.kda_state_alloc(cfg, 2)
    try:
        assert K.kda_state_max_slots(st) == 2
        assert K.kda_state_poll_error(st) == 0
    finally:
        K.kda_state_free(st)
    assert torch.cuda.mem_get_info()[0] >= free0 - (64 << 20)
