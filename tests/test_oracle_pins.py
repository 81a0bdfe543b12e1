"""The oracle's two forms (pure Python, scalar C) against the pins: values
fixed by the definition, hand-worked examples, closed forms, brute force over
the logical token stream, and the invariants the page states."""

import pytest

from helpers import FORMS
from pins import ALL_PINS


@pytest.mark.parametrize("form", sorted(FORMS))
@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, form):
    pin(FORMS[form])
