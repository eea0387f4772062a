# package marker
